"""GPU unmasked second-order operator (hla2_unmasked_forward, hla2_unmasked_step
through the C ABI) against the fp64 oracle: o_t = q_t^T S_t C_t (HLA summary,
section 1's naive product without the G correction)."""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_NORMALIZED, TOL_STEP_FP32, TOL_TC_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_FP32 = 1e-4  # CUDA-core walks, fp32 arithmetic from exact inputs


def tol(dtype, d, dv, norm):
    """Tensor-core walks (bf16 operands) get the bf16 bound, the CUDA-core
    walks the fp32 one, the normalised variant its own."""
    if norm:
        return TOL_NORMALIZED
    code = hla2.HLA2_DTYPE_BF16 if dtype == torch.bfloat16 else hla2.HLA2_DTYPE_F32
    return TOL_TC_BF16 if hla2.lib().hla2_unmasked_forward_path(d, dv, code, 0, 0) == 1 else TOL_FP32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def run_gpu(q, k, v, normalized=False, state_out=None):
    out = hla2.hla2_unmasked_forward(q.to(DEV), k.to(DEV), v.to(DEV), normalized=normalized, state_out=state_out)
    torch.cuda.synchronize()
    assert hla2.hla2_device_status() == 0
    return out


def inputs(B, H, T, d, dv, dtype, norm, seed):
    g = torch.Generator().manual_seed(seed)
    f = torch.rand if norm else torch.randn
    q = f(B, H, T, d, generator=g) / d ** 0.5
    k = f(B, H, T, d, generator=g) / d ** 0.5
    v = torch.randn(B, H, T, dv, generator=g) / (1.0 if norm else d ** 0.5)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def ref(q, k, v, normalized=False):
    return oracle.unmasked_serial(f64(q), f64(k), f64(v), normalized=normalized)


@pytest.mark.parametrize("B,H,T,d,dv,dtype,norm", [
    (1, 1, 1, 16, 16, torch.float32, False),
    (1, 2, 127, 64, 64, torch.bfloat16, False),
    (2, 1, 129, 64, 64, torch.bfloat16, False),
    (1, 3, 1000, 128, 128, torch.bfloat16, False),
    (1, 1, 700, 128, 64, torch.bfloat16, False),
    (1, 2, 300, 5, 3, torch.float32, False),
    (3, 1, 513, 64, 64, torch.bfloat16, True),
    (1, 1, 257, 128, 128, torch.float32, True),
    (1, 40, 200, 32, 32, torch.float32, False),
    (1, 2, 5000, 64, 64, torch.bfloat16, False),
])
def test_forward_shapes(B, H, T, d, dv, dtype, norm):
    q, k, v = inputs(B, H, T, d, dv, dtype, norm, seed=B * 1000 + H * 100 + T + d + 9)
    got = run_gpu(q, k, v, normalized=norm)
    assert relerr(f64(got), ref(q, k, v, norm)) < tol(dtype, d, dv, norm)


def test_tensor_core_path_selected():
    L = hla2.lib()
    assert L.hla2_unmasked_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_unmasked_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 0, 0) == 1
    assert L.hla2_unmasked_forward_path(64, 64, hla2.HLA2_DTYPE_BF16, 1, 0) == 0   # normalised: CUDA cores
    assert L.hla2_unmasked_forward_path(128, 128, hla2.HLA2_DTYPE_BF16, 0, 1) == 0  # state_out: CUDA cores
    assert L.hla2_unmasked_forward_path(128, 64, hla2.HLA2_DTYPE_BF16, 0, 0) == 0
    assert L.hla2_unmasked_forward_path(64, 64, hla2.HLA2_DTYPE_F32, 0, 0) == 0


@pytest.mark.parametrize("T", [1, 2, 3, 127, 128, 129, 383, 2000, 5000])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_walk_lengths(T, d):
    """Chunk boundaries, ragged tails, the split first chunk and multi-segment
    heads on the tcgen05 unmasked walks."""
    q, k, v = inputs(1, 3, T, d, d, torch.bfloat16, False, seed=T * 17 + d)
    got = run_gpu(q, k, v)
    assert relerr(f64(got), ref(q, k, v)) < TOL_TC_BF16


def test_tensor_core_matches_cuda_core_walk():
    """The tcgen05 walk and the fp32 CUDA-core walk (reached through
    state_out) agree on the same bf16 inputs within the bf16 bound."""
    q, k, v = inputs(2, 2, 1500, 128, 128, torch.bfloat16, False, seed=31)
    tc = run_gpu(q, k, v)
    st = torch.empty(4, hla2.unmasked_state_len(128, 128), device=DEV)
    cc = run_gpu(q, k, v, state_out=st)
    assert relerr(f64(tc), f64(cc)) < TOL_TC_BF16


def test_workload1_full():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w)
    assert relerr(f64(run_gpu(q, k, v)), ref(q, k, v)) < tol(q.dtype, w.d, w.dv, False)


def test_workload2_normalized_full():
    q, k, v = W.make_inputs(W.WORKLOADS[2])
    assert relerr(f64(run_gpu(q, k, v, normalized=True)), ref(q, k, v, True)) < TOL_NORMALIZED


def test_causality_bit_exact():
    q, k, v = inputs(1, 2, 1500, 64, 64, torch.bfloat16, False, seed=15)
    base = run_gpu(q, k, v)
    for cut in (0, 511, 1280):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        k2[..., cut + 1:, :] = -k2[..., cut + 1:, :]
        v2[..., cut + 1:, :] += 1
        assert torch.equal(run_gpu(q2, k2, v2)[..., :cut + 1, :], base[..., :cut + 1, :])


@pytest.mark.parametrize("norm", [False, True])
def test_state_out_then_step_continues(norm):
    B, H, T, extra, d, dv = 1, 3, 400, 20, 32, 32
    q, k, v = inputs(B, H, T + extra, d, dv, torch.float32, norm, seed=78)
    r = ref(q, k, v, norm)
    state = torch.empty(B * H, hla2.unmasked_state_len(d, dv), device=DEV)
    out = run_gpu(q[..., :T, :], k[..., :T, :], v[..., :T, :], normalized=norm, state_out=state)
    assert relerr(f64(out), r[..., :T, :]) < TOL_FP32
    kk, qq, vv = f64(k[..., :T, :])[0], f64(q[..., :T, :])[0], f64(v[..., :T, :])[0]
    expect = np.concatenate([np.einsum("hta,htb->hab", kk, kk).reshape(H, -1),
                             np.einsum("hta,hte->hae", qq, vv).reshape(H, -1), qq.sum(1)], axis=1)
    assert relerr(f64(state), expect) < 1e-5
    outs = []
    for t in range(T, T + extra):
        outs.append(hla2.hla2_unmasked_step(state, q[..., t, :].reshape(B * H, d).to(DEV),
                                            k[..., t, :].reshape(B * H, d).to(DEV),
                                            v[..., t, :].reshape(B * H, dv).to(DEV), normalized=norm))
    got = torch.stack(outs, dim=1).reshape(B, H, extra, dv)
    assert relerr(f64(got), r[..., T:, :]) < 1e-4


@pytest.mark.parametrize("d,dv,n,prefill,steps,norm", [(128, 128, 64, 64, 32, False), (64, 64, 33, 40, 16, True),
                                                       (4, 8, 3, 5, 7, False), (128, 32, 8, 8, 8, True)])
def test_step_from_shared_fp32_state(d, dv, n, prefill, steps, norm):
    w = W.DecodeWorkload("t", n, d, dv, prefill, steps, seed=13, normalized=norm)
    toks = list(W.decode_tokens(w))
    st = np.zeros((n, oracle.unmasked_state_len(d, dv)))
    for q, k, v in toks[:prefill]:
        st, _ = oracle.unmasked_step(st, f64(q), f64(k), f64(v), normalized=norm)
    st32 = st.astype(np.float32)
    st_ref = st32.astype(np.float64)
    st_gpu = torch.from_numpy(st32).to(DEV)
    for q, k, v in toks[prefill:]:
        st_ref, o_ref = oracle.unmasked_step(st_ref, f64(q), f64(k), f64(v), normalized=norm)
        o = hla2.hla2_unmasked_step(st_gpu, q.to(DEV), k.to(DEV), v.to(DEV), normalized=norm)
        assert relerr(f64(o), o_ref) < (TOL_NORMALIZED if norm else TOL_STEP_FP32)
    torch.cuda.synchronize()
    assert relerr(f64(st_gpu), st_ref) < 1e-5


def test_workload3_full_size_sampled_heads():
    """B1 H16 T65536 d=dv=128 (the benchmark's inputs and launch
    configuration): all heads on the GPU, three checked token by token."""
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    got = run_gpu(q, k, v)
    heads = [0, 8, 15]
    r = ref(q[:, heads], k[:, heads], v[:, heads])
    assert relerr(f64(got[:, heads]), r) < tol(q.dtype, w.d, w.dv, False)
    assert torch.isfinite(got).all()
