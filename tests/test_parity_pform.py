"""The compact P-form decode state (S | P = S C - G | p = S m - h):
hla2_step_pform and hla2_state_to_pform through the C ABI against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_NORMALIZED, TOL_STEP_FP32, f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


@pytest.mark.parametrize("d,dv,n,T", [(128, 128, 48, 40), (64, 64, 17, 33), (16, 16, 3, 20), (8, 32, 5, 9)])
def test_pform_steps_from_zero(d, dv, n, T):
    w = W.DecodeWorkload("t", n, d, dv, 0, T, seed=21)
    toks = list(W.decode_tokens(w))
    st = torch.zeros(n, hla2.pform_record_len(d, dv), device=DEV)
    got = [hla2.hla2_step_pform(st, q.to(DEV), k.to(DEV), v.to(DEV)) for q, k, v in toks]
    Q = np.stack([f64(t[0]) for t in toks], 1)  # [n, T, d]
    K = np.stack([f64(t[1]) for t in toks], 1)
    V = np.stack([f64(t[2]) for t in toks], 1)
    ref = oracle.serial(Q, K, V)
    assert relerr(np.stack([f64(o) for o in got], 1), ref) < TOL_STEP_FP32
    rec = oracle.chunk_summaries(Q, K, V, L=T)[:, 0]
    assert relerr(f64(st), oracle.summary_to_pform_state(rec, d, dv)) < TOL_STEP_FP32


def test_pform_normalized():
    d = dv = 64
    w = W.DecodeWorkload("t", 9, d, dv, 0, 25, seed=22, normalized=True)
    toks = list(W.decode_tokens(w))
    st = torch.zeros(9, hla2.pform_record_len(d, dv), device=DEV)
    got = [hla2.hla2_step_pform(st, q.to(DEV), k.to(DEV), v.to(DEV), normalized=True) for q, k, v in toks]
    Q = np.stack([f64(t[0]) for t in toks], 1)
    K = np.stack([f64(t[1]) for t in toks], 1)
    V = np.stack([f64(t[2]) for t in toks], 1)
    assert relerr(np.stack([f64(o) for o in got], 1), oracle.serial(Q, K, V, normalized=True)) < TOL_NORMALIZED


def test_state_to_pform_then_continue():
    """An fp32 G-form state (the oracle's prefill, rounded) converted on the GPU,
    then stepped in P-form, matches the oracle's continued recurrence."""
    d = dv = 128
    n, prefill, steps = 12, 30, 20
    w = W.DecodeWorkload("t", n, d, dv, prefill, steps, seed=23)
    toks = list(W.decode_tokens(w))
    st = np.zeros((n, oracle.record_len(d, dv)))
    for q, k, v in toks[:prefill]:
        st, _ = oracle.step(st, f64(q), f64(k), f64(v))
    st32 = st.astype(np.float32)
    g = torch.from_numpy(st32).to(DEV)
    pst = hla2.hla2_state_to_pform(g, d, dv)
    # expected conversion of the same fp32 state, in fp64
    S = st32[:, :d * d].astype(np.float64).reshape(n, d, d)
    C = st32[:, d * d:d * d + d * dv].astype(np.float64).reshape(n, d, dv)
    G = st32[:, d * d + d * dv:d * d + 2 * d * dv].astype(np.float64).reshape(n, d, dv)
    m = st32[:, d * d + 2 * d * dv:d * d + 2 * d * dv + d].astype(np.float64)
    h = st32[:, d * d + 2 * d * dv + d:].astype(np.float64)
    expect = np.concatenate([S.reshape(n, -1), (S @ C - G).reshape(n, -1), np.einsum("nab,nb->na", S, m) - h], 1)
    assert relerr(f64(pst), expect) < 1e-5
    ref_state = st32.astype(np.float64)
    got, ref = [], []
    for q, k, v in toks[prefill:]:
        ref_state, o = oracle.step(ref_state, f64(q), f64(k), f64(v))
        ref.append(o)
        got.append(hla2.hla2_step_pform(pst, q.to(DEV), k.to(DEV), v.to(DEV)))
    assert relerr(np.stack([f64(o) for o in got]), np.stack(ref)) < TOL_STEP_FP32


def test_pform_decode_workload_full_size_sampled_heads():
    """n=4096 heads, d=dv=128, 1024 + 512 tokens from a zero P-form state;
    eight heads checked on the last 512 outputs."""
    w = W.DECODE
    heads = [0, 5, 777, 2048, 4095]
    st = torch.zeros(w.n, hla2.pform_record_len(w.d, w.dv), device=DEV)
    sq, sk, sv, outs = [], [], [], []
    for t, (q, k, v) in enumerate(W.decode_tokens(w)):
        o = hla2.hla2_step_pform(st, q.to(DEV), k.to(DEV), v.to(DEV))
        sq.append(q[heads]); sk.append(k[heads]); sv.append(v[heads])
        if t >= w.prefill:
            outs.append(o[heads].cpu())
    Q = torch.stack(sq, 1)[:, None]
    K = torch.stack(sk, 1)[:, None]
    V = torch.stack(sv, 1)[:, None]
    ref = oracle.serial(f64(Q), f64(K), f64(V), nthreads=5)[:, 0, w.prefill:]
    assert relerr(torch.stack(outs, 1).double().numpy(), ref) < TOL_STEP_FP32
