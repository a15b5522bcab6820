"""GPU decayed masked operator (hla2_decay_forward, hla2_decay_step through the
C ABI) against the fp64 oracle:
o_t = sum_{i<=j<=t} gamma^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j.
Both sides take gamma as the same fp32 value."""
import numpy as np
import pytest
import torch

import oracle
from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_NORMALIZED, TOL_STEP_FP32, TOL_TC_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_FP32 = 1e-4  # CUDA-core walks and fp32 scan


def tol(dtype, d, dv, norm, gamma):
    """Tensor-core walks (bf16 operands) get the bf16 bound, the CUDA-core
    walks the fp32 one, the normalised variant its own."""
    if norm:
        return TOL_NORMALIZED
    code = hla2.HLA2_DTYPE_BF16 if dtype == torch.bfloat16 else hla2.HLA2_DTYPE_F32
    return TOL_TC_BF16 if hla2.lib().hla2_decay_forward_path(d, dv, code, 0, 0, gamma) == 1 else TOL_FP32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def g32(g):
    return float(np.float32(g))


def run_gpu(q, k, v, gamma, normalized=False, state_out=None):
    out = hla2.hla2_decay_forward(q.to(DEV), k.to(DEV), v.to(DEV), gamma, normalized=normalized, state_out=state_out)
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


def ref(q, k, v, gamma, normalized=False):
    return oracle.decay_serial(f64(q), f64(k), f64(v), g32(gamma), normalized=normalized)


@pytest.mark.parametrize("gamma", [0.999, 0.9, 0.5])
@pytest.mark.parametrize("B,H,T,d,dv,dtype,norm", [
    (1, 1, 1, 16, 16, torch.float32, False),
    (1, 2, 300, 64, 64, torch.bfloat16, False),
    (1, 3, 1000, 128, 128, torch.bfloat16, False),
    (1, 1, 700, 128, 64, torch.bfloat16, False),
    (1, 2, 300, 5, 3, torch.float32, False),
    (3, 1, 513, 64, 64, torch.bfloat16, True),
    (1, 40, 200, 32, 32, torch.float32, False),
    (1, 2, 5000, 64, 64, torch.bfloat16, False),
])
def test_forward_shapes(B, H, T, d, dv, dtype, norm, gamma):
    q, k, v = inputs(B, H, T, d, dv, dtype, norm, seed=B * 1000 + H * 100 + T + d + 11)
    got = run_gpu(q, k, v, g32(gamma), normalized=norm)
    assert relerr(f64(got), ref(q, k, v, gamma, norm)) < tol(dtype, d, dv, norm, g32(gamma))


def test_tensor_core_path_selected():
    L = hla2.lib()
    bf = hla2.HLA2_DTYPE_BF16
    assert L.hla2_decay_forward_path(128, 128, bf, 0, 0, g32(0.999)) == 1
    assert L.hla2_decay_forward_path(64, 64, bf, 0, 0, 1.0) == 1
    assert L.hla2_decay_forward_path(64, 64, bf, 0, 0, 0.8) == 1
    assert L.hla2_decay_forward_path(64, 64, bf, 0, 0, g32(0.79)) == 0   # below the tensor-core range
    assert L.hla2_decay_forward_path(64, 64, bf, 1, 0, g32(0.99)) == 0   # normalised: CUDA cores
    assert L.hla2_decay_forward_path(128, 128, bf, 0, 1, g32(0.99)) == 0  # state_out: CUDA cores
    assert L.hla2_decay_forward_path(128, 64, bf, 0, 0, g32(0.99)) == 0
    assert L.hla2_decay_forward_path(64, 64, hla2.HLA2_DTYPE_F32, 0, 0, g32(0.99)) == 0


@pytest.mark.parametrize("gamma", [1.0, 0.999, 0.95, 0.8])
@pytest.mark.parametrize("T", [1, 2, 127, 129, 383, 2000, 5000])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_walk_lengths(T, d, gamma):
    """Chunk boundaries, ragged tails, the split first chunk, multi-segment
    heads and the ends of the tensor-core gamma range on the tcgen05 walks."""
    q, k, v = inputs(1, 3, T, d, d, torch.bfloat16, False, seed=T * 19 + d)
    got = run_gpu(q, k, v, g32(gamma))
    assert relerr(f64(got), ref(q, k, v, g32(gamma))) < TOL_TC_BF16


def test_tensor_core_matches_cuda_core_walk():
    """The tcgen05 walk and the fp32 CUDA-core walk (reached through
    state_out) agree on the same bf16 inputs within the bf16 bound."""
    q, k, v = inputs(2, 2, 1500, 128, 128, torch.bfloat16, False, seed=32)
    gamma = g32(0.97)
    tc = run_gpu(q, k, v, gamma)
    st = torch.empty(4, hla2.pform_record_len(128, 128), device=DEV)
    cc = run_gpu(q, k, v, gamma, state_out=st)
    assert relerr(f64(tc), f64(cc)) < TOL_TC_BF16


def test_gamma_one_matches_the_masked_oracle():
    q, k, v = inputs(1, 2, 2000, 64, 64, torch.bfloat16, False, seed=3)
    got = run_gpu(q, k, v, 1.0)
    assert relerr(f64(got), oracle.serial(f64(q), f64(k), f64(v))) < tol(q.dtype, 64, 64, False, 1.0)


def test_workload1_full():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w)
    assert relerr(f64(run_gpu(q, k, v, g32(0.999))), ref(q, k, v, 0.999)) < tol(q.dtype, w.d, w.dv, False, g32(0.999))


def test_causality_bit_exact():
    q, k, v = inputs(1, 2, 1500, 64, 64, torch.bfloat16, False, seed=16)
    base = run_gpu(q, k, v, g32(0.95))
    for cut in (0, 700, 1280):
        k2, v2 = k.clone(), v.clone()
        k2[..., cut + 1:, :] = -k2[..., cut + 1:, :]
        v2[..., cut + 1:, :] += 1
        assert torch.equal(run_gpu(q, k2, v2, g32(0.95))[..., :cut + 1, :], base[..., :cut + 1, :])


def test_rejects_bad_gamma():
    q = torch.zeros(1, 1, 8, 16, device=DEV)
    with pytest.raises(hla2.HLA2Error):
        hla2.hla2_decay_forward(q, q, q, 1.5)
    s = torch.zeros(2, hla2.pform_record_len(16, 16), device=DEV)
    x = torch.zeros(2, 16, device=DEV)
    with pytest.raises(hla2.HLA2Error):
        hla2.hla2_decay_step(s, x, x, x, -0.1)


@pytest.mark.parametrize("norm", [False, True])
def test_state_out_then_step_continues(norm):
    B, H, T, extra, d, dv = 1, 3, 400, 20, 32, 32
    gamma = g32(0.97)
    q, k, v = inputs(B, H, T + extra, d, dv, torch.float32, norm, seed=79)
    r = ref(q, k, v, gamma, norm)
    state = torch.empty(B * H, hla2.pform_record_len(d, dv), device=DEV)
    out = run_gpu(q[..., :T, :], k[..., :T, :], v[..., :T, :], gamma, normalized=norm, state_out=state)
    assert relerr(f64(out), r[..., :T, :]) < TOL_FP32
    summ = oracle.decay_chunk_summaries(f64(q[..., :T, :]), f64(k[..., :T, :]), f64(v[..., :T, :]), T, gamma)[:, :, 0]
    expect = oracle.summary_to_pform_state(summ, d, dv).reshape(B * H, -1)
    assert relerr(f64(state), expect) < 1e-5
    outs = []
    for t in range(T, T + extra):
        outs.append(hla2.hla2_decay_step(state, q[..., t, :].reshape(B * H, d).to(DEV),
                                         k[..., t, :].reshape(B * H, d).to(DEV),
                                         v[..., t, :].reshape(B * H, dv).to(DEV), gamma, normalized=norm))
    got = torch.stack(outs, dim=1).reshape(B, H, extra, dv)
    assert relerr(f64(got), r[..., T:, :]) < 1e-4


@pytest.mark.parametrize("d,dv,n,prefill,steps,norm,gamma", [(128, 128, 64, 64, 32, False, 0.99),
                                                             (64, 64, 33, 40, 16, True, 0.9),
                                                             (4, 8, 3, 5, 7, False, 0.5)])
def test_step_from_shared_fp32_state(d, dv, n, prefill, steps, norm, gamma):
    gamma = g32(gamma)
    w = W.DecodeWorkload("t", n, d, dv, prefill, steps, seed=14, normalized=norm)
    toks = list(W.decode_tokens(w))
    st = np.zeros((n, d * d + d * dv + d))
    for q, k, v in toks[:prefill]:
        st, _ = oracle.decay_step_pform(st, f64(q), f64(k), f64(v), gamma, norm)
    st32 = st.astype(np.float32)
    st_ref = st32.astype(np.float64)
    st_gpu = torch.from_numpy(st32).to(DEV)
    for q, k, v in toks[prefill:]:
        st_ref, o_ref = oracle.decay_step_pform(st_ref, f64(q), f64(k), f64(v), gamma, norm)
        o = hla2.hla2_decay_step(st_gpu, q.to(DEV), k.to(DEV), v.to(DEV), gamma, normalized=norm)
        assert relerr(f64(o), o_ref) < (TOL_NORMALIZED if norm else TOL_STEP_FP32)
    torch.cuda.synchronize()
    assert relerr(f64(st_gpu), st_ref) < 1e-5


def test_workload3_full_size_sampled_heads():
    """B1 H16 T65536 d=dv=128 with gamma = 0.999 (the benchmark's decayed
    line): all heads on the GPU, three checked token by token."""
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    gamma = g32(0.999)
    got = run_gpu(q, k, v, gamma)
    heads = [0, 8, 15]
    r = ref(q[:, heads], k[:, heads], v[:, heads], gamma)
    assert relerr(f64(got[:, heads]), r) < tol(q.dtype, w.d, w.dv, False, gamma)
    assert torch.isfinite(got).all()
