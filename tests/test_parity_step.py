"""GPU decode step (hla2_step through the C ABI) against the fp64 oracle."""
import time

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


def oracle_prefill_state(toks, d, dv):
    """fp64 oracle state after the prefill tokens, rounded to fp32 (the shared
    starting point of both sides)."""
    n = toks[0][0].shape[0]
    state = np.zeros((n, oracle.record_len(d, dv)))
    for q, k, v in toks:
        state, _ = oracle.step(state, f64(q), f64(k), f64(v))
    return state.astype(np.float32)


@pytest.mark.parametrize("d,dv,n,prefill,steps", [(128, 128, 64, 64, 32), (64, 64, 33, 40, 16),
                                                  (16, 16, 5, 10, 10), (4, 8, 3, 5, 7), (128, 32, 8, 8, 8)])
def test_step_from_shared_fp32_state(d, dv, n, prefill, steps):
    w = W.DecodeWorkload("t", n, d, dv, prefill, steps, seed=11)
    toks = list(W.decode_tokens(w))
    st32 = oracle_prefill_state(toks[:prefill], d, dv)
    st_ref = st32.astype(np.float64)
    st_gpu = torch.from_numpy(st32).to(DEV)
    outs_ref, outs_gpu = [], []
    for q, k, v in toks[prefill:]:
        st_ref, o = oracle.step(st_ref, f64(q), f64(k), f64(v))
        outs_ref.append(o)
        outs_gpu.append(hla2.hla2_step(st_gpu, q.to(DEV), k.to(DEV), v.to(DEV)))
    torch.cuda.synchronize()
    assert relerr(np.stack([f64(o) for o in outs_gpu]), np.stack(outs_ref)) < TOL_STEP_FP32
    assert relerr(f64(st_gpu), st_ref) < TOL_STEP_FP32


def test_step_normalized():
    d = dv = 64
    w = W.DecodeWorkload("t", 16, d, dv, 30, 30, seed=12, normalized=True)
    toks = list(W.decode_tokens(w))
    st_ref = np.zeros((16, oracle.record_len(d, dv)))
    st_gpu = torch.zeros(16, oracle.record_len(d, dv), device=DEV)
    ref, got = [], []
    for q, k, v in toks:
        st_ref, o = oracle.step(st_ref, f64(q), f64(k), f64(v), normalized=True)
        ref.append(o)
        got.append(hla2.hla2_step(st_gpu, q.to(DEV), k.to(DEV), v.to(DEV), normalized=True))
    assert relerr(np.stack([f64(o) for o in got]), np.stack(ref)) < TOL_NORMALIZED


def test_decode_workload_full_size_sampled_heads():
    """n=4096 heads, d=dv=128: the GPU prefills every head with 1024 steps from
    a zero state, then takes the 512 timed-size steps; eight heads are checked
    on all 512 outputs against the oracle's fp64 recurrence over all 1536
    tokens."""
    w = W.DECODE
    heads = [0, 1, 511, 1024, 2047, 3000, 4094, 4095]
    st = torch.zeros(w.n, W.state_floats(w.d, w.dv), device=DEV)
    sq, sk, sv, outs = [], [], [], []
    for t, (q, k, v) in enumerate(W.decode_tokens(w)):
        o = hla2.hla2_step(st, q.to(DEV, non_blocking=True), k.to(DEV, non_blocking=True),
                           v.to(DEV, non_blocking=True))
        sq.append(q[heads]); sk.append(k[heads]); sv.append(v[heads])
        if t >= w.prefill:
            outs.append(o[heads].cpu())
    Q = torch.stack(sq, 1)[:, None]  # [heads, 1, T, d] -> oracle heads axis
    K = torch.stack(sk, 1)[:, None]
    V = torch.stack(sv, 1)[:, None]
    ref = oracle.serial(f64(Q), f64(K), f64(V), nthreads=8)[:, 0, w.prefill:]
    got = torch.stack(outs, 1).double().numpy()
    assert relerr(got, ref) < TOL_STEP_FP32


def test_step_cost_independent_of_prefix():
    """Per-token cost does not depend on the prefix length: a step on a state
    that has absorbed 4096 tokens takes as long as one on a fresh state."""
    n, d = 2048, 128
    R = W.state_floats(d, d)
    fresh = torch.zeros(n, R, device=DEV)
    long = torch.zeros(n, R, device=DEV)
    q = torch.randn(n, d, device=DEV) / d ** 0.5
    for _ in range(64):  # put non-zero, grown values in `long`
        hla2.hla2_step(long, q, q, q)
    long.mul_(64.0)

    def timeit(st):
        for _ in range(3):
            hla2.hla2_step(st, q, q, q)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            hla2.hla2_step(st, q, q, q)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    a, b = timeit(fresh), timeit(long)
    assert 0.7 < a / b < 1.4
