"""GPU forward (hla2_forward through the C ABI) against the fp64 oracle.

Inputs are the seeded workloads; sizes span several 128-token chunks,
several segments and ragged tails.  Full-size workloads are compared on
every head where the oracle finishes in seconds, otherwise on sampled heads
(all of their tokens).
"""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import (TOL_FP32_WALK, TOL_NORMALIZED, TOL_TC_BF16, f64, forward_tolerance, oracle_forward,
                           relerr, NTHREADS)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_gpu(q, k, v, normalized=False, state_out=None):
    out = hla2.hla2_forward(q.to(DEV), k.to(DEV), v.to(DEV), normalized=normalized, state_out=state_out)
    torch.cuda.synchronize()
    assert hla2.hla2_device_status() == 0
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def test_tensor_core_path_selected():
    """bf16 d = dv in {64, 128} (unnormalised) runs on the tcgen05 walks; the
    other cases run on the CUDA-core walks.  Both are this library's kernels."""
    L = hla2.lib()
    assert L.hla2_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 1, 0) == 1   # normalised: split operands
    assert L.hla2_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 1, 0) == 0
    assert L.hla2_forward_path(16, 16, hla2.HLA2_DTYPE_F32, 0, 0) == 0
    # the final state is handed over from the tensor-core forward too
    assert L.hla2_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 1) == 1
    assert L.hla2_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 0, 1) == 1
    assert L.hla2_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 1, 1) == 1


@pytest.mark.parametrize("T", [1, 127, 128, 129, 383, 2000, 5000])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_walk_lengths(T, d):
    """Chunk boundaries, ragged tails and multi-segment heads on the tcgen05 walks."""
    g = torch.Generator().manual_seed(T * 7 + d)
    B, H = 1, 3
    q = (torch.randn(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    k = (torch.randn(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    v = (torch.randn(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), oracle_forward(q, k, v)) < TOL_TC_BF16


@pytest.mark.parametrize("T", [1, 127, 128, 129, 1000, 3000])
def test_tensor_core_normalized_lengths(T):
    """Ratio-normalised variant on the tcgen05 walks (d = 64, split operands)."""
    d = 64
    g = torch.Generator().manual_seed(T * 11 + 5)
    B, H = 2, 2
    q = (torch.rand(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    k = (torch.rand(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    v = torch.randn(B, H, T, d, generator=g).to(torch.bfloat16)
    got = run_gpu(q, k, v, normalized=True)
    assert relerr(f64(got), oracle_forward(q, k, v, normalized=True)) < TOL_NORMALIZED


# ------------------------------------------------------ seeded workloads ----
def test_workload0_fp32_d16():
    w = W.WORKLOADS[0]
    q, k, v = W.make_inputs(w)
    ref = oracle_forward(q, k, v)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), ref) < TOL_FP32_WALK


def test_workload1_full():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w)
    ref = oracle_forward(q, k, v)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), ref) < TOL_TC_BF16


def test_workload2_normalized_full():
    w = W.WORKLOADS[2]
    q, k, v = W.make_inputs(w)
    ref = oracle_forward(q, k, v, normalized=True)
    got = run_gpu(q, k, v, normalized=True)
    assert relerr(f64(got), ref) < TOL_NORMALIZED


def test_workload3_full_size_sampled_heads():
    """B1 H16 T65536 d=dv=128: all heads run on the GPU in the benchmark's
    launch configuration; three heads are checked token by token."""
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    got = run_gpu(q, k, v)
    heads = [0, 7, 15]
    ref = oracle.serial(f64(q[:, heads]), f64(k[:, heads]), f64(v[:, heads]), nthreads=3)
    assert relerr(f64(got[:, heads]), ref) < TOL_TC_BF16
    assert torch.isfinite(got).all()


def test_workload3_recipe_short_all_heads():
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w, T=3000)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), oracle_forward(q, k, v)) < TOL_TC_BF16


# ------------------------------------------------------------ edge cases ----
@pytest.mark.parametrize("B,H,T,d,dv,dtype,norm", [
    (1, 1, 1, 16, 16, torch.float32, False),      # single token
    (1, 2, 127, 64, 64, torch.bfloat16, False),   # one ragged chunk
    (2, 1, 129, 64, 64, torch.bfloat16, False),   # chunk + 1
    (1, 3, 1000, 128, 128, torch.bfloat16, False),
    (1, 1, 700, 128, 64, torch.bfloat16, False),  # d != dv
    (1, 2, 300, 5, 3, torch.float32, False),      # odd sizes
    (1, 1, 50, 1, 1, torch.float32, False),       # scalar case
    (3, 1, 513, 64, 64, torch.bfloat16, True),    # normalised, ragged
    (1, 1, 257, 128, 128, torch.float32, True),
    (1, 40, 200, 32, 32, torch.float32, False),   # many heads, short
])
def test_edge_shapes(B, H, T, d, dv, dtype, norm):
    g = torch.Generator().manual_seed(B * 1000 + H * 100 + T + d)
    if norm:
        q = torch.rand(B, H, T, d, generator=g) / d ** 0.5
        k = torch.rand(B, H, T, d, generator=g) / d ** 0.5
        v = torch.randn(B, H, T, dv, generator=g)
    else:
        q = torch.randn(B, H, T, d, generator=g) / d ** 0.5
        k = torch.randn(B, H, T, d, generator=g) / d ** 0.5
        v = torch.randn(B, H, T, dv, generator=g) / d ** 0.5
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    got = run_gpu(q, k, v, normalized=norm)
    ref = oracle_forward(q, k, v, normalized=norm)
    assert relerr(f64(got), ref) < forward_tolerance(dtype, d, dv, norm)


def test_zero_inputs_give_zero():
    q = torch.zeros(1, 2, 300, 64, dtype=torch.bfloat16)
    got = run_gpu(q, q, torch.zeros(1, 2, 300, 64, dtype=torch.bfloat16))
    assert (got == 0).all()


# ------------------------------------------------------------ invariants ----
def test_causality_bit_exact_on_gpu():
    """Perturbing tokens after t leaves every output at or before t unchanged."""
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w, B=1, H=4, T=1500)
    base = run_gpu(q, k, v)
    for cut in (0, 200, 777, 1280):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[..., cut + 1:, :] = -q2[..., cut + 1:, :] * 2
        k2[..., cut + 1:, :] = k2[..., cut + 1:, :].flip(-1)
        v2[..., cut + 1:, :] += 1
        out = run_gpu(q2, k2, v2)
        assert torch.equal(out[..., :cut + 1, :], base[..., :cut + 1, :]), cut


def test_deterministic():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w, B=1, H=4, T=1100)
    a = run_gpu(q, k, v)
    b = run_gpu(q, k, v)
    assert torch.equal(a, b)


def test_zero_padding_within_tolerance():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w, B=1, H=2, T=900)
    pad = lambda x: torch.cat([x, torch.zeros(*x.shape[:2], 300, x.shape[-1], dtype=x.dtype)], dim=2)
    a = run_gpu(q, k, v)
    b = run_gpu(pad(q), pad(k), pad(v))[..., :900, :]
    assert relerr(f64(b), f64(a)) < 1e-3


# -------------------------------------------------- prefill -> decode -----
@pytest.mark.parametrize("dtype,norm", [(torch.float32, False), (torch.bfloat16, False), (torch.float32, True)])
def test_state_out_then_step_continues(dtype, norm):
    """forward(T) hands its final state to hla2_step; stepping the next tokens
    reproduces the oracle's outputs for the whole sequence."""
    B, H, T, extra, d, dv = 1, 3, 400, 20, 32, 32
    g = torch.Generator().manual_seed(77)
    if norm:
        q = torch.rand(B, H, T + extra, d, generator=g) / d ** 0.5
        k = torch.rand(B, H, T + extra, d, generator=g) / d ** 0.5
    else:
        q = torch.randn(B, H, T + extra, d, generator=g) / d ** 0.5
        k = torch.randn(B, H, T + extra, d, generator=g) / d ** 0.5
    v = torch.randn(B, H, T + extra, dv, generator=g) / d ** 0.5
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    ref = oracle_forward(q, k, v, normalized=norm)
    state = torch.empty(B * H, hla2.record_len(d, dv), device=DEV)
    out = run_gpu(q[..., :T, :], k[..., :T, :], v[..., :T, :], normalized=norm, state_out=state)
    assert relerr(f64(out), ref[..., :T, :]) < TOL_FP32_WALK
    # the handed-over state equals the oracle's whole-prefix summary
    summ = oracle.chunk_summaries(f64(q[..., :T, :]), f64(k[..., :T, :]), f64(v[..., :T, :]), L=T)[:, :, 0]
    expect = oracle.summary_to_decode_state(summ, d, dv).reshape(B * H, -1)
    assert relerr(f64(state), expect) < 1e-5
    outs = []
    for t in range(T, T + extra):
        qt = q[..., t, :].reshape(B * H, d).float().to(DEV)
        kt = k[..., t, :].reshape(B * H, d).float().to(DEV)
        vt = v[..., t, :].reshape(B * H, dv).float().to(DEV)
        outs.append(hla2.hla2_step(state, qt, kt, vt, normalized=norm))
    got = torch.stack(outs, dim=1).reshape(B, H, extra, dv)
    assert relerr(f64(got), ref[..., T:, :]) < 1e-4


@pytest.mark.parametrize("d,T,norm", [(128, 129, False), (128, 1000, False), (128, 3000, False),
                                      (64, 129, False), (64, 1000, False), (64, 3000, False),
                                      (64, 1000, True), (64, 3000, True)])
def test_state_out_tensor_core(d, T, norm):
    """bf16 d = dv in {64, 128} with state_out on the tcgen05 walks (one-chunk
    segments with a one-token tail at T = 129, a scan short enough for one
    launch at T = 1000, a longer one at T = 3000): S, C and m of the handed-over
    state are fp32 sums (1e-5 per field); G and h carry the walks' rounding
    (the forward's bound over the whole state); decoding then continues."""
    assert hla2.lib().hla2_forward_path(d, d, hla2.HLA2_DTYPE_BF16, int(norm), 1) == 1
    B, H, extra, dv = 1, 3, 12, d
    g = torch.Generator().manual_seed(d * 1000 + T + int(norm))
    if norm:
        q = torch.rand(B, H, T + extra, d, generator=g) / d ** 0.5
        k = torch.rand(B, H, T + extra, d, generator=g) / d ** 0.5
    else:
        q = torch.randn(B, H, T + extra, d, generator=g) / d ** 0.5
        k = torch.randn(B, H, T + extra, d, generator=g) / d ** 0.5
    v = torch.randn(B, H, T + extra, dv, generator=g) / d ** 0.5
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    tol = TOL_NORMALIZED if norm else TOL_TC_BF16
    ref = oracle_forward(q, k, v, normalized=norm)
    state = torch.empty(B * H, hla2.record_len(d, dv), device=DEV)
    out = run_gpu(q[..., :T, :], k[..., :T, :], v[..., :T, :], normalized=norm, state_out=state)
    assert relerr(f64(out), ref[..., :T, :]) < tol
    summ = oracle.chunk_summaries(f64(q[..., :T, :]), f64(k[..., :T, :]), f64(v[..., :T, :]), L=T)[:, :, 0]
    expect = oracle.summary_to_decode_state(summ, d, dv).reshape(B * H, -1)
    got = f64(state)
    nS, nC = d * d, d * dv
    cut = {"S": (0, nS), "C": (nS, nS + nC), "m": (nS + 2 * nC, nS + 2 * nC + d)}
    for name, (a, b) in cut.items():
        assert relerr(got[:, a:b], expect[:, a:b]) < 1e-5, name
    assert relerr(got, expect) < tol
    outs = []
    for t in range(T, T + extra):
        qt = q[..., t, :].reshape(B * H, d).float().to(DEV)
        kt = k[..., t, :].reshape(B * H, d).float().to(DEV)
        vt = v[..., t, :].reshape(B * H, dv).float().to(DEV)
        outs.append(hla2.hla2_step(state, qt, kt, vt, normalized=norm))
    got_o = torch.stack(outs, dim=1).reshape(B, H, extra, dv)
    assert relerr(f64(got_o), ref[..., T:, :]) < tol


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_state_out_graph_capture(dtype):
    """The forward with state_out issues only stream-ordered work too: captured
    in a CUDA graph and replayed on new inputs it gives the eager O and final
    state bit for bit."""
    B, H, T, d = 1, 4, 2000, 64 if dtype == torch.bfloat16 else 32
    g0 = torch.Generator().manual_seed(5)
    mk = lambda: [(torch.randn(B, H, T, d, generator=g0) / d ** 0.5).to(dtype).to(DEV) for _ in range(3)]
    (q, k, v), (q2, k2, v2) = mk(), mk()
    ws = torch.empty(hla2.hla2_forward_workspace(B, H, T, d, d, hla2.HLA2_DTYPE_BF16 if dtype == torch.bfloat16
                                                 else hla2.HLA2_DTYPE_F32), device=DEV, dtype=torch.uint8)
    O = torch.empty(B, H, T, d, device=DEV)
    st = torch.empty(B * H, hla2.record_len(d, d), device=DEV)
    call = lambda a, b, c: hla2.hla2_forward(a, b, c, O, workspace=ws, state_out=st)
    refs = []
    for x in ((q2, k2, v2), (q, k, v)):
        call(*x)
        torch.cuda.synchronize()
        refs.append((O.clone(), st.clone()))
    sq, sk, sv = q.clone(), k.clone(), v.clone()
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        call(sq, sk, sv)
        cs.synchronize()
        with torch.cuda.graph(graph, stream=cs):
            call(sq, sk, sv)
    torch.cuda.synchronize()
    for (a, b, c), (o_ref, s_ref) in (((q, k, v), refs[1]), ((q2, k2, v2), refs[0])):
        sq.copy_(a); sk.copy_(b); sv.copy_(c)
        O.zero_(); st.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(O, o_ref)
        assert torch.equal(st, s_ref)
    assert hla2.hla2_device_status() == 0


@pytest.mark.parametrize("op", ["hla", "ahla", "unmasked", "decay"])
def test_cuda_graph_replay_matches_eager(op):
    """The forwards issue only stream-ordered work (no allocation, no host
    synchronisation), so they can be captured in a CUDA graph: replays on new
    inputs give the eager results bit for bit."""
    calls = {"hla": lambda q, k, v, O, ws: hla2.hla2_forward(q, k, v, O, workspace=ws),
             "ahla": lambda q, k, v, O, ws: hla2.hla2_ahla_forward(q, k, v, O, workspace=ws),
             "unmasked": lambda q, k, v, O, ws: hla2.hla2_unmasked_forward(q, k, v, O, workspace=ws),
             "decay": lambda q, k, v, O, ws: hla2.hla2_decay_forward(q, k, v, 0.99, O, workspace=ws)}
    call = calls[op]
    w = W.WORKLOADS[1]
    q, k, v = (x.to(DEV) for x in W.make_inputs(w))
    q2, k2, v2 = (x.to(DEV) for x in W.make_inputs(w, seed=77))
    ws = torch.empty(hla2.hla2_forward_workspace(w.B, w.H, w.T, w.d, w.dv, hla2.HLA2_DTYPE_BF16),
                     device=DEV, dtype=torch.uint8)
    O = torch.empty(w.B, w.H, w.T, w.dv, device=DEV)
    call(q2, k2, v2, O, ws)
    ref2 = O.clone()
    call(q, k, v, O, ws)
    ref1 = O.clone()
    sq, sk, sv = q.clone(), k.clone(), v.clone()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        call(sq, sk, sv, O, ws)
        cs.synchronize()
        with torch.cuda.graph(g, stream=cs):
            call(sq, sk, sv, O, ws)
    torch.cuda.synchronize()
    O.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O, ref1)
    sq.copy_(q2); sk.copy_(k2); sv.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O, ref2)
    assert hla2.hla2_device_status() == 0
