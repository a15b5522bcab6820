"""GPU AHLA (hla2_ahla_forward, hla2_ahla_step through the C ABI) against the
fp64 oracle (HLA summary, section 2 "AHLA").

The forward runs segment summaries, the exclusive scan with the semidirect
combine (M_B P_A cross term) and segment walks; sizes span several
128-token chunks, several segments per head and ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_NORMALIZED, TOL_STEP_FP32, TOL_TC_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# CUDA-core AHLA walks: fp32 arithmetic from exact inputs.
TOL_AHLA_FP32 = 1e-4


def tol(dtype, d, dv, norm):
    """Tensor-core walks (bf16 operands) get the bf16 bound, the CUDA-core
    walks the fp32 one, the normalised variant its own."""
    if norm:
        return TOL_NORMALIZED
    code = hla2.HLA2_DTYPE_BF16 if dtype == torch.bfloat16 else hla2.HLA2_DTYPE_F32
    return TOL_TC_BF16 if hla2.lib().hla2_ahla_forward_path(d, dv, code, 0, 0) == 1 else TOL_AHLA_FP32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def run_gpu(q, k, v, normalized=False, state_out=None):
    out = hla2.hla2_ahla_forward(q.to(DEV), k.to(DEV), v.to(DEV), normalized=normalized, state_out=state_out)
    torch.cuda.synchronize()
    assert hla2.hla2_device_status() == 0
    return out


def inputs(B, H, T, d, dv, dtype, norm, seed):
    g = torch.Generator().manual_seed(seed)
    if norm:
        q = torch.rand(B, H, T, d, generator=g) / d ** 0.5
        k = torch.rand(B, H, T, d, generator=g) / d ** 0.5
        v = torch.randn(B, H, T, dv, generator=g)
    else:
        q = torch.randn(B, H, T, d, generator=g) / d ** 0.5
        k = torch.randn(B, H, T, d, generator=g) / d ** 0.5
        v = torch.randn(B, H, T, dv, generator=g) / d ** 0.5
    return q.to(dtype), k.to(dtype), v.to(dtype)


def ref(q, k, v, normalized=False):
    return oracle.ahla_serial(f64(q), f64(k), f64(v), normalized=normalized)


@pytest.mark.parametrize("B,H,T,d,dv,dtype,norm", [
    (1, 1, 1, 16, 16, torch.float32, False),      # single token
    (1, 2, 127, 64, 64, torch.bfloat16, False),   # one ragged chunk
    (2, 1, 129, 64, 64, torch.bfloat16, False),   # chunk + 1
    (1, 3, 1000, 128, 128, torch.bfloat16, False),
    (1, 1, 700, 128, 64, torch.bfloat16, False),  # d != dv
    (1, 1, 700, 32, 128, torch.float32, False),   # d < dv
    (1, 2, 300, 5, 3, torch.float32, False),      # odd sizes
    (1, 1, 50, 1, 1, torch.float32, False),       # scalar case
    (3, 1, 513, 64, 64, torch.bfloat16, True),    # normalised, ragged
    (1, 1, 257, 128, 128, torch.float32, True),
    (1, 40, 200, 32, 32, torch.float32, False),   # many heads, short
    (1, 2, 5000, 64, 64, torch.bfloat16, False),  # many segments per head
])
def test_forward_shapes(B, H, T, d, dv, dtype, norm):
    q, k, v = inputs(B, H, T, d, dv, dtype, norm, seed=B * 1000 + H * 100 + T + d + 7)
    got = run_gpu(q, k, v, normalized=norm)
    assert relerr(f64(got), ref(q, k, v, norm)) < tol(dtype, d, dv, norm)


def test_tensor_core_path_selected():
    L = hla2.lib()
    assert L.hla2_ahla_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_ahla_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_ahla_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 1, 0) == 0   # normalised: CUDA cores
    assert L.hla2_ahla_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 1) == 0  # state_out: CUDA cores
    assert L.hla2_ahla_forward_path(128, 64, hla2.HLA2_DTYPE_BF16, 0, 0) == 0
    assert L.hla2_ahla_forward_path(64, 64, hla2.HLA2_DTYPE_F32, 0, 0) == 0


@pytest.mark.parametrize("T", [1, 2, 3, 127, 128, 129, 383, 2000, 5000])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_walk_lengths(T, d):
    """Chunk boundaries, ragged tails, the split first chunk and multi-segment
    heads on the tcgen05 AHLA walks."""
    q, k, v = inputs(1, 3, T, d, d, torch.bfloat16, False, seed=T * 13 + d)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), ref(q, k, v)) < TOL_TC_BF16


def test_tensor_core_matches_cuda_core_path():
    """The same bf16 inputs through both implementations (state_out selects
    the CUDA-core walks)."""
    B, H, T, d = 1, 4, 3000, 128
    q, k, v = inputs(B, H, T, d, d, torch.bfloat16, False, seed=41)
    tc = run_gpu(q, k, v)
    st = torch.empty(B * H, hla2.ahla_state_len(d, d), device=DEV)
    cc = run_gpu(q, k, v, state_out=st)
    assert relerr(f64(tc), f64(cc)) < TOL_TC_BF16


def test_workload1_full():
    """B2 H8 T2048 d=dv=64 bf16 inputs, every head token by token."""
    q, k, v = W.make_inputs(W.WORKLOADS[1])
    assert relerr(f64(run_gpu(q, k, v)), ref(q, k, v)) < tol(torch.bfloat16, 64, 64, False)


def test_workload2_normalized_full():
    """B4 H16 T4096 d=dv=64, uniform q, k: the ratio-normalised variant."""
    w = W.WORKLOADS[2]
    q, k, v = W.make_inputs(w)
    got = run_gpu(q, k, v, normalized=True)
    assert relerr(f64(got), ref(q, k, v, True)) < TOL_NORMALIZED


def test_workload3_full_size_sampled_heads():
    """B1 H16 T65536 d=dv=128: all heads on the GPU, two checked by the oracle."""
    q, k, v = W.make_inputs(W.WORKLOADS[3])
    got = run_gpu(q, k, v)
    heads = [0, 11]
    r = ref(q[:, heads], k[:, heads], v[:, heads])
    assert relerr(f64(got[:, heads]), r) < tol(torch.bfloat16, 128, 128, False)
    assert torch.isfinite(got).all()


def test_causality_bit_exact():
    q, k, v = inputs(1, 3, 1500, 64, 64, torch.bfloat16, False, seed=5)
    base = run_gpu(q, k, v)
    for cut in (0, 200, 777, 1280):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[..., cut + 1:, :] = -q2[..., cut + 1:, :] * 2
        k2[..., cut + 1:, :] = k2[..., cut + 1:, :].flip(-1)
        v2[..., cut + 1:, :] += 1
        out = run_gpu(q2, k2, v2)
        assert torch.equal(out[..., :cut + 1, :], base[..., :cut + 1, :]), cut


def test_deterministic_and_zero():
    q, k, v = inputs(1, 2, 1100, 64, 64, torch.bfloat16, False, seed=6)
    assert torch.equal(run_gpu(q, k, v), run_gpu(q, k, v))
    z = torch.zeros(1, 2, 300, 64, dtype=torch.bfloat16)
    assert (run_gpu(z, z, z) == 0).all()


@pytest.mark.parametrize("norm", [False, True])
def test_state_out_then_step_continues(norm):
    """The forward's final P|E|m|n equals the oracle's whole-prefix summary;
    hla2_ahla_step continues the sequence from it."""
    B, H, T, extra, d, dv = 1, 3, 400, 20, 32, 32
    q, k, v = inputs(B, H, T + extra, d, dv, torch.float32, norm, seed=77)
    r = ref(q, k, v, norm)
    state = torch.empty(B * H, hla2.ahla_state_len(d, dv), device=DEV)
    out = run_gpu(q[..., :T, :], k[..., :T, :], v[..., :T, :], normalized=norm, state_out=state)
    assert relerr(f64(out), r[..., :T, :]) < TOL_AHLA_FP32
    summ = oracle.ahla_chunk_summaries(f64(q[..., :T, :]), f64(k[..., :T, :]), f64(v[..., :T, :]), L=T)[:, :, 0]
    expect = oracle.ahla_summary_to_state(summ, d, dv).reshape(B * H, -1)
    assert relerr(f64(state), expect) < 1e-5
    outs = []
    for t in range(T, T + extra):
        qt = q[..., t, :].reshape(B * H, d).to(DEV)
        kt = k[..., t, :].reshape(B * H, d).to(DEV)
        vt = v[..., t, :].reshape(B * H, dv).to(DEV)
        outs.append(hla2.hla2_ahla_step(state, qt, kt, vt, normalized=norm))
    got = torch.stack(outs, dim=1).reshape(B, H, extra, dv)
    assert relerr(f64(got), r[..., T:, :]) < 1e-4


@pytest.mark.parametrize("d,dv,n,prefill,steps,norm", [(128, 128, 64, 64, 32, False), (64, 64, 33, 40, 16, True),
                                                       (16, 16, 5, 10, 10, False), (4, 8, 3, 5, 7, True),
                                                       (128, 32, 8, 8, 8, False)])
def test_step_from_shared_fp32_state(d, dv, n, prefill, steps, norm):
    """Both sides start from the same fp32 state (the oracle's prefill,
    rounded) and take the same tokens; every output is compared."""
    w = W.DecodeWorkload("t", n, d, dv, prefill, steps, seed=12, normalized=norm)
    toks = list(W.decode_tokens(w))
    st = np.zeros((n, oracle.ahla_state_len(d, dv)))
    for q, k, v in toks[:prefill]:
        st, _ = oracle.ahla_step(st, f64(q), f64(k), f64(v), normalized=norm)
    st32 = st.astype(np.float32)
    st_ref = st32.astype(np.float64)
    st_gpu = torch.from_numpy(st32).to(DEV)
    for q, k, v in toks[prefill:]:
        st_ref, o_ref = oracle.ahla_step(st_ref, f64(q), f64(k), f64(v), normalized=norm)
        o = hla2.hla2_ahla_step(st_gpu, q.to(DEV), k.to(DEV), v.to(DEV), normalized=norm)
        tol = TOL_NORMALIZED if norm else TOL_STEP_FP32
        assert relerr(f64(o), o_ref) < tol
    torch.cuda.synchronize()
    assert relerr(f64(st_gpu), st_ref) < 1e-5


def test_step_rejects_bad_sizes():
    s = torch.zeros(2, hla2.ahla_state_len(12, 12), device=DEV)
    q = torch.zeros(2, 12, device=DEV)
    with pytest.raises(hla2.HLA2Error):
        hla2.hla2_ahla_step(s, q, q, q)
