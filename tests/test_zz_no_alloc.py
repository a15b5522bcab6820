"""hla2_forward_noalloc: the forward for callers that cannot allocate device
scratch (for example a host framework that owns a fixed device arena and
forbids cudaMalloc inside its callbacks).  The library then uses its own
fixed-size static device array.  This file is collected last, so a run that
stops at the first failure has already run every other test.

Checks, through the C ABI: two calls in a row match hla2_forward (with a
caller workspace) within the parity tolerances, on the tensor-core path and
on the CUDA-core path; a problem needing more than the fixed array is
rejected with a clear message and leaves the output untouched."""
import ctypes

import pytest
import torch

from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_FP32_WALK, TOL_TC_BF16, f64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CAPACITY = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def _noalloc_raw(q, k, v, o, normalized=False):
    """Call the C entry point directly (no Python-side allocation)."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    L = hla2.lib()
    return L.hla2_forward_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                  ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                  B, H, T, d, dv, int(normalized),
                                  hla2.HLA2_DTYPE_BF16 if q.dtype == torch.bfloat16 else hla2.HLA2_DTYPE_F32,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["tensor_core_bf16_d128", "cuda_core_normalized_fp32_d64"])
def test_noalloc_matches_forward_twice(case):
    if case == "tensor_core_bf16_d128":
        w = W.WORKLOADS[3]
        q, k, v = (x.to(DEV) for x in W.make_inputs(w, H=4, T=3000))
        norm, tol = False, TOL_TC_BF16
    else:
        w = W.WORKLOADS[2]
        q, k, v = (x.float().to(DEV) for x in W.make_inputs(w, B=1, H=2, T=777))
        norm, tol = True, TOL_FP32_WALK
    B, H, T, d = q.shape
    need = hla2.hla2_forward_workspace(B, H, T, d, v.shape[-1],
                                       hla2.HLA2_DTYPE_BF16 if q.dtype == torch.bfloat16 else hla2.HLA2_DTYPE_F32)
    assert 0 < need <= CAPACITY
    ref = hla2.hla2_forward(q, k, v, normalized=norm)
    for _ in range(2):  # the array keeps the previous call's contents; the result must not depend on them
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc_raw(q, k, v, out, normalized=norm)
        assert rc == hla2.HLA2_OK, hla2.hla2_last_error_detail()
        torch.cuda.synchronize()
        assert hla2.hla2_device_status() == 0
        assert torch.isfinite(out).all()
        assert relerr(f64(out), f64(ref)) < tol


def test_noalloc_rejects_problems_beyond_capacity():
    """The smallest head count (T = 16384, d = dv = 128) whose scratch exceeds
    the fixed array is rejected with a message naming the size; O is untouched."""
    B, T, d = 1, 16384, 128
    H = next(h for h in (16, 32, 64, 128, 256, 512)
             if hla2.hla2_forward_workspace(B, h, T, d, d, hla2.HLA2_DTYPE_BF16) > CAPACITY)
    need = hla2.hla2_forward_workspace(B, H, T, d, d, hla2.HLA2_DTYPE_BF16)
    assert need > CAPACITY
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device=DEV)
    o = torch.full((B, H, T, d), 7.0, device=DEV)
    rc = _noalloc_raw(q, q, q, o)
    assert rc == hla2.HLA2_ERR_UNSUPPORTED
    msg = hla2.hla2_last_error_detail()
    assert "scratch" in msg and str(need) in msg
    torch.cuda.synchronize()
    assert (o == 7.0).all()
    with pytest.raises(hla2.HLA2Error):
        hla2.hla2_forward_noalloc(q, q, q, o)


def test_noalloc_wrapper_rejects_bad_arguments_before_launch():
    """The Python wrapper checks what the C entry point cannot see (it only
    gets pointers): an O of the wrong shape, and Q, K, V of mixed dtypes
    (fp32 Q with bf16 K would make the kernels read K past its end).  Both
    raise before anything is launched, so O keeps its contents."""
    w = W.WORKLOADS[1]
    q, k, v = (x.to(DEV) for x in W.make_inputs(w, B=1, H=2, T=300))
    B, H, T, _ = q.shape
    dv = v.shape[-1]
    small = torch.full((B, H, T - 1, dv), 7.0, device=DEV)
    with pytest.raises(ValueError, match="shape"):
        hla2.hla2_forward_noalloc(q, k, v, O=small)
    o = torch.full((B, H, T, dv), 7.0, device=DEV)
    with pytest.raises(ValueError, match="share a dtype"):
        hla2.hla2_forward_noalloc(q.float(), k, v, O=o)
    torch.cuda.synchronize()
    assert (small == 7.0).all() and (o == 7.0).all()


def test_noalloc_writes_stay_inside_o():
    """O is carved out of a larger allocation whose margins hold a byte
    pattern; after two calls (T = 129 and a ragged 5000) every margin byte
    still holds it, and the inputs are unchanged."""
    margin = 64 * 1024
    w = W.WORKLOADS[3]
    for T in (129, 5000):
        q, k, v = (x.to(DEV) for x in W.make_inputs(w, H=3, T=T))
        B, H, _, d = q.shape
        dv = v.shape[-1]
        n = B * H * T * dv
        buf = torch.empty(n + 2 * (margin // 4), device=DEV, dtype=torch.float32)
        buf.view(torch.uint8).fill_(0xA5)
        o = buf[margin // 4: margin // 4 + n].view(B, H, T, dv)
        snap = [x.clone() for x in (q, k, v)]
        rc = _noalloc_raw(q, k, v, o)
        assert rc == hla2.HLA2_OK, hla2.hla2_last_error_detail()
        torch.cuda.synchronize()
        assert hla2.hla2_device_status() == 0
        b = buf.view(torch.uint8)
        assert (b[:margin] == 0xA5).all() and (b[margin + 4 * n:] == 0xA5).all()
        assert all(torch.equal(x, y) for x, y in zip((q, k, v), snap))
        assert torch.isfinite(o).all()
