"""GPU chunk summaries and exclusive scan (hla2_chunk_summaries, hla2_scan)
against the fp64 oracle's definitions."""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def per_field_err(got, ref, d, dv):
    """Relative error per record field (S, C, m, G, h), each scaled by its own max."""
    nS, nC = d * d, d * dv
    cuts = [0, nS, nS + nC, nS + nC + d, nS + 2 * nC + d, nS + 2 * nC + 2 * d]
    return [relerr(got[..., a:b], ref[..., a:b]) for a, b in zip(cuts[:-1], cuts[1:])]


@pytest.mark.parametrize("wid,L,B,H,T", [(0, 16, None, None, None), (1, 64, 1, 3, 1000), (3, 64, 1, 2, 1300),
                                          (0, 7, None, None, 61)])
def test_chunk_summaries(wid, L, B, H, T):
    w = W.WORKLOADS[wid]
    q, k, v = W.make_inputs(w, B=B, H=H, T=T)
    got = hla2.hla2_chunk_summaries(q.to(DEV), k.to(DEV), v.to(DEV), L)
    ref = oracle.chunk_summaries(f64(q), f64(k), f64(v), L=L)
    assert max(per_field_err(f64(got), ref, w.d, w.dv)) < 1e-5


@pytest.mark.parametrize("d,dv,N,BH", [(16, 16, 4, 1), (64, 64, 32, 3), (128, 128, 9, 2), (5, 3, 17, 2)])
def test_scan_matches_oracle_fold(d, dv, N, BH):
    """Same fp32 summaries in; the oracle folds the combine left to right."""
    rng = np.random.default_rng(d * 100 + N)
    T = N * 8
    Q = rng.standard_normal((BH, T, d)) / np.sqrt(d)
    K = rng.standard_normal((BH, T, d)) / np.sqrt(d)
    V = rng.standard_normal((BH, T, dv)) / np.sqrt(d)
    summ = oracle.chunk_summaries(Q, K, V, L=8).astype(np.float32)
    ref = oracle.scan_fold(summ.astype(np.float64), d, dv)
    got = hla2.hla2_scan(torch.from_numpy(summ).reshape(1, BH, N, -1).to(DEV), d, dv)
    errs = per_field_err(f64(got).reshape(BH, N, -1)[:, 1:], ref[:, 1:], d, dv)
    assert max(errs) < 1e-5, errs
    assert (got[:, :, 0] == 0).all()


def test_summaries_then_scan_restart_equals_serial_state():
    """GPU summaries -> GPU scan: prefix n equals the oracle state after n chunks."""
    w = W.WORKLOADS[1]
    L = 64
    q, k, v = W.make_inputs(w, B=1, H=2, T=64 * 12)
    s = hla2.hla2_chunk_summaries(q.to(DEV), k.to(DEV), v.to(DEV), L)
    p = hla2.hla2_scan(s, w.d, w.dv)
    for n in (1, 5, 11):
        ref = oracle.chunk_summaries(f64(q[..., :n * L, :]), f64(k[..., :n * L, :]), f64(v[..., :n * L, :]),
                                     L=n * L)[..., 0, :]
        errs = per_field_err(f64(p[..., n, :]), ref, w.d, w.dv)
        assert max(errs) < 1e-5, (n, errs)


def test_scan_long_context_chunk_level():
    """1024 chunks of 64 at d=dv=128 (one head of the long-context workload):
    GPU summaries and scan against the oracle's summaries and fold."""
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w, H=1)
    s = hla2.hla2_chunk_summaries(q.to(DEV), k.to(DEV), v.to(DEV), 64)
    p = hla2.hla2_scan(s, w.d, w.dv)
    ref_s = oracle.chunk_summaries(f64(q), f64(k), f64(v), L=64)
    assert max(per_field_err(f64(s), ref_s, w.d, w.dv)) < 1e-5
    ref_p = oracle.scan_fold(ref_s[0, 0], w.d, w.dv)
    errs = per_field_err(f64(p[0, 0, 1:]), ref_p[1:], w.d, w.dv)
    assert max(errs) < 1e-4, errs


@pytest.mark.parametrize("d,L,T", [(64, 64, 1000), (64, 128, 1000), (128, 64, 777), (128, 128, 640),
                                   (128, 64, 64), (64, 64, 65), (128, 128, 1)])
def test_chunk_summaries_tensor_core(d, L, T):
    """bf16 inputs with d = dv in {64, 128} and L in {64, 128} take the
    tensor-core kernel (two chunks per 128-token tile at L = 64; odd chunk
    counts and ragged tails leave the missing chunk unwritten); every field
    stays within the fp32 walk's 1e-5 of the oracle."""
    assert hla2.lib().hla2_chunk_summaries_path(d, d, L, hla2.HLA2_DTYPE_BF16) == 1
    assert hla2.lib().hla2_chunk_summaries_path(d, d, 32, hla2.HLA2_DTYPE_BF16) == 0
    assert hla2.lib().hla2_chunk_summaries_path(d, d, L, hla2.HLA2_DTYPE_F32) == 0
    g = torch.Generator().manual_seed(d + L + T)
    B, H = 1, 3
    q, k, v = ((torch.randn(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16) for _ in range(3))
    got = hla2.hla2_chunk_summaries(q.to(DEV), k.to(DEV), v.to(DEV), L)
    ref = oracle.chunk_summaries(f64(q), f64(k), f64(v), L=L)
    errs = per_field_err(f64(got), ref, d, d)
    assert max(errs) < 1e-5, errs
