"""Thin Python binding of libhla2 (the C ABI in include/hla2.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks type/shape/contiguity, and passes raw device pointers,
sizes and the current CUDA stream to the C entry point of the same name.  All
computation happens in the library's CUDA kernels.  If ``libhla2.so`` is
missing or cannot be loaded, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhla2.so")

HLA2_OK = 0
HLA2_ERR_INVALID = -1
HLA2_ERR_UNSUPPORTED = -2
HLA2_ERR_WORKSPACE = -3
HLA2_ERR_LAUNCH = -4
HLA2_ERR_DEVICE = -5
HLA2_DTYPE_F32 = 0
HLA2_DTYPE_BF16 = 1

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class HLA2Error(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where} failed with status {code}: {detail}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libhla2.so (built in-tree by ``higher_order_linear_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libhla2.so not built ({LIB_PATH}); run higher_order_linear_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.hla2_forward_workspace.argtypes = [i, i, i, i, i, i]
            L.hla2_forward_workspace.restype = sz
            L.hla2_forward_plan.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i)]
            L.hla2_forward_plan.restype = i
            L.hla2_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp, vp]
            L.hla2_forward.restype = i
            L.hla2_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
            L.hla2_step.restype = i
            L.hla2_chunk_summaries.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
            L.hla2_chunk_summaries.restype = i
            L.hla2_scan.argtypes = [vp, vp, i, i, i, i, i, vp]
            L.hla2_scan.restype = i
            L.hla2_last_error_detail.argtypes = [ctypes.c_char_p, sz]
            L.hla2_last_error_detail.restype = i
            L.hla2_device_status.argtypes = [vp]
            L.hla2_device_status.restype = i
            L.hla2_selftest_wait_runout.argtypes = [vp, i, vp]
            L.hla2_selftest_wait_runout.restype = i
            L.hla2_profile_enable.argtypes = [i]
            L.hla2_profile_enable.restype = i
            L.hla2_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), i, ctypes.POINTER(i),
                                            ctypes.POINTER(ctypes.c_longlong)]
            L.hla2_profile_read.restype = i
            L.hla2_forward_path.argtypes = [i, i, i, i, i]
            L.hla2_forward_path.restype = i
            L.hla2_chunk_summaries_path.argtypes = [i, i, i, i]
            L.hla2_chunk_summaries_path.restype = i
            L.hla2_forward_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
            L.hla2_forward_noalloc.restype = i
            L.hla2_forward_host_workspace.argtypes = [i, i, i, i, i, i, i]
            L.hla2_forward_host_workspace.restype = sz
            L.hla2_forward_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, sz, vp]
            L.hla2_forward_host.restype = i
            L.hla2_step_pform.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
            L.hla2_step_pform.restype = i
            L.hla2_state_to_pform.argtypes = [vp, vp, i, i, i, vp]
            L.hla2_state_to_pform.restype = i
            L.hla2_ahla_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp, vp]
            L.hla2_ahla_forward.restype = i
            L.hla2_ahla_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
            L.hla2_ahla_step.restype = i
            L.hla2_ahla_forward_path.argtypes = [i, i, i, i, i]
            L.hla2_ahla_forward_path.restype = i
            L.hla2_unmasked_forward_path.argtypes = [i, i, i, i, i]
            L.hla2_unmasked_forward_path.restype = i
            L.hla2_decay_forward_path.argtypes = [i, i, i, i, i, ctypes.c_float]
            L.hla2_decay_forward_path.restype = i
            L.hla2_unmasked_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp, vp]
            L.hla2_unmasked_forward.restype = i
            L.hla2_unmasked_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
            L.hla2_unmasked_step.restype = i
            L.hla2_decay_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, vp, sz, vp, vp]
            L.hla2_decay_forward.restype = i
            L.hla2_decay_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, vp]
            L.hla2_decay_step.restype = i
            _lib = L
        return _lib


def hla2_last_error_detail() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().hla2_last_error_detail(buf, 512)
    return buf.value.decode(errors="replace")


def _check(code: int, where: str) -> None:
    if code != HLA2_OK:
        raise HLA2Error(code, where, hla2_last_error_detail())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return HLA2_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return HLA2_DTYPE_BF16
    raise ValueError(f"unsupported input dtype {t.dtype}")


def _same_device(device: torch.device, **tensors) -> None:
    """Every tensor must live on ``device`` (the first input's): the library
    launches on the current device, which the calls below make ``device``."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the inputs on {device}")


def _qkv(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor):
    """Shape, dtype and device checks shared by the forwards; returns
    (B, H, T, d, dv, dtype code).  Runs before anything touches the library."""
    if Q.dim() != 4 or K.shape != Q.shape or V.dim() != 4 or V.shape[:3] != Q.shape[:3]:
        raise ValueError("expected Q, K [B,H,T,d] and V [B,H,T,dv]")
    if not (Q.dtype == K.dtype == V.dtype):
        raise ValueError(f"Q, K, V must share a dtype (got {Q.dtype}, {K.dtype}, {V.dtype})")
    _same_device(Q.device, K=K, V=V)
    B, H, T, d = Q.shape
    return B, H, T, d, V.shape[-1], _dtype_code(Q)


def _out(O: torch.Tensor | None, shape, device: torch.device) -> torch.Tensor:
    """The caller's output tensor, checked, or a new fp32 one."""
    if O is None:
        return torch.empty(shape, device=device, dtype=torch.float32)
    if tuple(O.shape) != tuple(shape):
        raise ValueError(f"O has shape {tuple(O.shape)}, expected {tuple(shape)}")
    if O.dtype != torch.float32:
        raise ValueError(f"O must be float32, got {O.dtype}")
    if not O.is_contiguous():
        raise ValueError("O must be contiguous")
    _same_device(device, O=O)
    return O


def hla2_forward_workspace(B: int, H: int, T: int, d: int, dv: int, dtype: int) -> int:
    return int(lib().hla2_forward_workspace(B, H, T, d, dv, dtype))


def hla2_forward_plan(B: int, H: int, T: int, sm_count: int = 0):
    """The forward's segment plan: (segments per head, chunks of 128 tokens
    per segment, SM count planned for).  sm_count <= 0 plans for the current
    device, as hla2_forward does."""
    ns, ln, used = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().hla2_forward_plan(B, H, T, int(sm_count), ctypes.byref(ns), ctypes.byref(ln), ctypes.byref(used)),
           "hla2_forward_plan")
    return int(ns.value), int(ln.value), int(used.value)


def record_len(d: int, dv: int) -> int:
    return d * d + 2 * d * dv + 2 * d


def _cuda_device(t: torch.Tensor, name: str) -> torch.device:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.device


def _forward(entry: str, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None,
             normalized: bool, workspace: torch.Tensor | None, state_out: torch.Tensor | None, stream,
             state_len: int | None, gamma: float | None = None) -> torch.Tensor:
    """Common marshalling of the four forwards (same C signature, plus gamma
    before the dtype for the decayed one).  Every check runs before the
    library is touched; the call itself runs with Q's device current, so the
    default stream and the library's per-device state are that device's."""
    B, H, T, d, dv, code = _qkv(Q, K, V)
    O = _out(O, (B, H, T, dv), Q.device)
    if state_out is not None:
        if state_len is None or state_out.numel() != B * H * state_len:
            raise ValueError(f"state_out must hold B*H = {B * H} states of {state_len} floats")
    _same_device(Q.device, workspace=workspace, state_out=state_out)
    dev = _cuda_device(Q, "Q")
    with torch.cuda.device(dev):
        need = hla2_forward_workspace(B, H, T, d, dv, code)
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
        sptr = _dev(state_out, "state_out", torch.float32) if state_out is not None else None
        args = [_dev(Q, "Q"), _dev(K, "K"), _dev(V, "V"), _dev(O, "O", torch.float32),
                B, H, T, d, dv, int(bool(normalized))]
        if gamma is not None:
            args.append(float(gamma))
        args += [code, _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), sptr,
                 _stream(stream)]
        rc = getattr(lib(), entry)(*args)
    _check(rc, entry)
    return O


def hla2_forward(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                 normalized: bool = False, workspace: torch.Tensor | None = None,
                 state_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Masked second-order HLA forward.  Q, K [B,H,T,d], V [B,H,T,dv] (fp32 or
    bf16, same dtype, same device) -> O [B,H,T,dv] fp32.  ``state_out``
    [B*H, record] fp32 receives the final decode state S|C|G|m|h if given."""
    return _forward("hla2_forward", Q, K, V, O, normalized, workspace, state_out, stream, record_len(*_dims(Q, V)))


def _dims(Q: torch.Tensor, V: torch.Tensor):
    return (Q.shape[-1] if Q.dim() else 0), (V.shape[-1] if V.dim() else 0)


def hla2_forward_noalloc(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                         normalized: bool = False, stream=None) -> torch.Tensor:
    """hla2_forward for callers that cannot allocate device scratch: the
    library uses its own fixed 64 MiB device array instead of a workspace
    (larger problems raise).  Only O is allocated here, and only when the
    caller passes none.  The arguments are checked as for hla2_forward
    before anything is launched."""
    B, H, T, d, dv, code = _qkv(Q, K, V)
    O = _out(O, (B, H, T, dv), Q.device)
    dev = _cuda_device(Q, "Q")
    with torch.cuda.device(dev):
        rc = lib().hla2_forward_noalloc(_dev(Q, "Q"), _dev(K, "K"), _dev(V, "V"), _dev(O, "O", torch.float32),
                                        B, H, T, d, dv, int(bool(normalized)), code, _stream(stream))
    _check(rc, "hla2_forward_noalloc")
    return O


def _host(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def hla2_forward_host_workspace(B: int, H: int, T: int, d: int, dv: int, dtype: int, heads_per_group: int = 0) -> int:
    return int(lib().hla2_forward_host_workspace(B, H, T, d, dv, dtype, heads_per_group))


def hla2_forward_host(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                      normalized: bool = False, heads_per_group: int = 0, dev: torch.Tensor | None = None,
                      stream=None, device=None) -> torch.Tensor:
    """Masked forward on host tensors (pinned for overlap): Q, K [B,H,T,d],
    V [B,H,T,dv] on the CPU -> O [B,H,T,dv] fp32 on the CPU.  The library
    copies groups of heads in, runs the forward and copies O out as a
    pipeline on the GPU that holds ``dev`` (else ``device``, else the current
    one), which is made current for the call; O is complete once ``stream``
    (that device's current stream by default) has been synchronised.  ``dev``
    is the device buffer of hla2_forward_host_workspace(...) bytes (allocated
    here when None)."""
    if Q.dim() != 4 or K.shape != Q.shape or V.dim() != 4 or V.shape[:3] != Q.shape[:3]:
        raise ValueError("expected Q, K [B,H,T,d] and V [B,H,T,dv]")
    if not (Q.dtype == K.dtype == V.dtype):
        raise ValueError("Q, K, V must share a dtype")
    B, H, T, d = Q.shape
    dv = V.shape[-1]
    code = _dtype_code(Q)
    if O is None:
        O = torch.empty((B, H, T, dv), dtype=torch.float32, pin_memory=Q.is_pinned())
    elif O.shape != (B, H, T, dv):
        raise ValueError("O has the wrong shape")
    if dev is not None:
        gpu = _cuda_device(dev, "dev")
        if device is not None and torch.device(device) != gpu:
            raise ValueError(f"dev is on {gpu}, device is {device}")
    else:
        gpu = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(gpu):
        need = hla2_forward_host_workspace(B, H, T, d, dv, code, heads_per_group)
        if dev is None:
            dev = torch.empty(max(need, 256), dtype=torch.uint8, device=gpu)
        rc = lib().hla2_forward_host(_host(Q, "Q"), _host(K, "K"), _host(V, "V"), _host(O, "O", torch.float32),
                                     B, H, T, d, dv, int(bool(normalized)), code, int(heads_per_group),
                                     _dev(dev, "dev"), dev.numel() * dev.element_size(), _stream(stream))
    _check(rc, "hla2_forward_host")
    return O


def _step(entry: str, state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
          o: torch.Tensor | None, normalized: bool, stream, state_len_fn, gamma: float | None = None) -> torch.Tensor:
    """Common marshalling of the decode steps: state [n, state_len] fp32
    (updated in place), q, k [n, d], v [n, dv] fp32 -> o [n, dv] fp32."""
    if q.dim() != 2 or k.shape != q.shape or v.dim() != 2 or v.shape[0] != q.shape[0]:
        raise ValueError(f"{entry}: expected q, k [n,d] and v [n,dv]")
    n, d = q.shape
    dv = v.shape[-1]
    if state.numel() != n * state_len_fn(d, dv):
        raise ValueError(f"{entry}: state must hold n = {n} states of {state_len_fn(d, dv)} floats")
    if o is not None and tuple(o.shape) != (n, dv):
        raise ValueError(f"{entry}: o has shape {tuple(o.shape)}, expected {(n, dv)}")
    _same_device(q.device, k=k, v=v, state=state, o=o)
    dev = _cuda_device(q, "q")
    with torch.cuda.device(dev):
        if o is None:
            o = torch.empty((n, dv), device=dev, dtype=torch.float32)
        args = [_dev(state, "state", torch.float32), _dev(q, "q", torch.float32), _dev(k, "k", torch.float32),
                _dev(v, "v", torch.float32), _dev(o, "o", torch.float32), n, d, dv, int(bool(normalized))]
        if gamma is not None:
            args.append(float(gamma))
        args.append(_stream(stream))
        rc = getattr(lib(), entry)(*args)
    _check(rc, entry)
    return o


def hla2_step(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
              o: torch.Tensor | None = None, normalized: bool = False, stream=None) -> torch.Tensor:
    """One decode step for n heads.  state [n, record] fp32 (S|C|G|m|h,
    updated in place), q, k [n, d], v [n, dv] fp32 -> o [n, dv] fp32."""
    return _step("hla2_step", state, q, k, v, o, normalized, stream, record_len)


def pform_record_len(d: int, dv: int) -> int:
    return d * d + d * dv + d


def hla2_step_pform(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    o: torch.Tensor | None = None, normalized: bool = False, stream=None) -> torch.Tensor:
    """Decode step on the compact P-form state [n, d*d + d*dv + d] (S | P | p)."""
    return _step("hla2_step_pform", state, q, k, v, o, normalized, stream, pform_record_len)


def hla2_state_to_pform(gstate: torch.Tensor, d: int, dv: int, pstate: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """S|C|G|m|h decode states -> S|P|p (P = S C - G, p = S m - h)."""
    n = gstate.numel() // record_len(d, dv)
    if gstate.numel() != n * record_len(d, dv):
        raise ValueError("gstate size is not a whole number of records")
    if pstate is not None and pstate.numel() != n * pform_record_len(d, dv):
        raise ValueError(f"pstate must hold n = {n} states of {pform_record_len(d, dv)} floats")
    _same_device(gstate.device, pstate=pstate)
    dev = _cuda_device(gstate, "gstate")
    with torch.cuda.device(dev):
        if pstate is None:
            pstate = torch.empty((n, pform_record_len(d, dv)), device=dev, dtype=torch.float32)
        rc = lib().hla2_state_to_pform(_dev(gstate, "gstate", torch.float32), _dev(pstate, "pstate", torch.float32),
                                       n, d, dv, _stream(stream))
    _check(rc, "hla2_state_to_pform")
    return pstate


def hla2_chunk_summaries(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, L: int,
                         summ: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """[B,H,N,record] fp32 chunk summaries S|C|m|G|h, N = ceil(T/L)."""
    B, H, T, d, dv, code = _qkv(Q, K, V)
    if L <= 0:
        raise ValueError("chunk length L must be positive")
    N = (T + L - 1) // L
    if summ is not None and summ.numel() != B * H * N * record_len(d, dv):
        raise ValueError(f"summ must hold B*H*N = {B * H * N} records of {record_len(d, dv)} floats")
    _same_device(Q.device, summ=summ)
    dev = _cuda_device(Q, "Q")
    with torch.cuda.device(dev):
        if summ is None:
            summ = torch.empty((B, H, N, record_len(d, dv)), device=dev, dtype=torch.float32)
        rc = lib().hla2_chunk_summaries(_dev(Q, "Q"), _dev(K, "K"), _dev(V, "V"), _dev(summ, "summ", torch.float32),
                                        B, H, T, d, dv, int(L), code, _stream(stream))
    _check(rc, "hla2_chunk_summaries")
    return summ


def hla2_scan(summ: torch.Tensor, d: int, dv: int, prefix: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exclusive scan of [B,H,N,record] summaries with the semidirect combine."""
    if summ.dim() != 4:
        raise ValueError("summ must be [B,H,N,record]")
    B, H, N, R = summ.shape
    if R != record_len(d, dv):
        raise ValueError("record length does not match d, dv")
    if prefix is not None and tuple(prefix.shape) != tuple(summ.shape):
        raise ValueError("prefix must have the shape of summ")
    _same_device(summ.device, prefix=prefix)
    dev = _cuda_device(summ, "summ")
    with torch.cuda.device(dev):
        if prefix is None:
            prefix = torch.empty_like(summ)
        rc = lib().hla2_scan(_dev(summ, "summ", torch.float32), _dev(prefix, "prefix", torch.float32),
                             B, H, N, d, dv, _stream(stream))
    _check(rc, "hla2_scan")
    return prefix


def hla2_device_status(stream=None) -> int:
    return int(lib().hla2_device_status(_stream(stream)))


def hla2_selftest_wait_runout(flag: torch.Tensor, wait_us: int, stream=None) -> None:
    """Runs the library's wait run-out on purpose (see include/hla2.h); flag
    is a CUDA int32 tensor of one element that receives 0 when the wait gave
    up.  Read the status afterwards with hla2_device_status."""
    if not (isinstance(flag, torch.Tensor) and flag.is_cuda and flag.dtype == torch.int32 and flag.numel() >= 1):
        raise ValueError("flag must be a CUDA int32 tensor with at least one element")
    with torch.cuda.device(flag.device):
        _check(lib().hla2_selftest_wait_runout(ctypes.c_void_p(flag.data_ptr()), int(wait_us), _stream(stream)),
               "hla2_selftest_wait_runout")


def hla2_profile_enable(on: bool = True) -> None:
    _check(lib().hla2_profile_enable(int(bool(on))), "hla2_profile_enable")


def hla2_profile_read():
    """(phase_ms[3], profiled forwards, kernels launched) since the last read;
    phases are segment summaries, scan, segment outputs."""
    ms = (ctypes.c_float * 3)()
    nf = ctypes.c_int(0)
    nl = ctypes.c_longlong(0)
    _check(lib().hla2_profile_read(ms, 3, ctypes.byref(nf), ctypes.byref(nl)), "hla2_profile_read")
    return [float(x) for x in ms], int(nf.value), int(nl.value)


# ------------------------------------------------------------------ AHLA ----
def ahla_state_len(d: int, dv: int) -> int:
    """AHLA decode state per head: P (d x dv) | E (d x dv) | m (d) | n (d)."""
    return 2 * d * dv + 2 * d


def hla2_ahla_forward(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                      normalized: bool = False, workspace: torch.Tensor | None = None,
                      state_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Masked AHLA forward (o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j).
    Shapes and dtypes as for hla2_forward; ``state_out`` [B*H, 2*d*dv + 2*d]
    fp32 receives the final P|E|m|n state if given."""
    return _forward("hla2_ahla_forward", Q, K, V, O, normalized, workspace, state_out, stream,
                    ahla_state_len(*_dims(Q, V)))


def hla2_ahla_step(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                   o: torch.Tensor | None = None, normalized: bool = False, stream=None) -> torch.Tensor:
    """One AHLA decode step for n heads: state [n, 2*d*dv + 2*d] fp32 (P|E|m|n,
    updated in place), q, k [n, d], v [n, dv] fp32 -> o [n, dv] fp32."""
    return _step("hla2_ahla_step", state, q, k, v, o, normalized, stream, ahla_state_len)


# -------------------------------------------------------------- unmasked ----
def unmasked_state_len(d: int, dv: int) -> int:
    """Unmasked decode state per head: S (d x d) | C (d x dv) | m (d)."""
    return d * d + d * dv + d


def hla2_unmasked_forward(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                          normalized: bool = False, workspace: torch.Tensor | None = None,
                          state_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Unmasked second-order forward o_t = q_t^T S_t C_t.  Shapes and dtypes
    as for hla2_forward; ``state_out`` [B*H, d*d + d*dv + d] fp32 receives the
    final S|C|m if given."""
    return _forward("hla2_unmasked_forward", Q, K, V, O, normalized, workspace, state_out, stream,
                    unmasked_state_len(*_dims(Q, V)))


def hla2_unmasked_step(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       o: torch.Tensor | None = None, normalized: bool = False, stream=None) -> torch.Tensor:
    """One unmasked decode step: state [n, d*d + d*dv + d] fp32 (S|C|m, in place)."""
    return _step("hla2_unmasked_step", state, q, k, v, o, normalized, stream, unmasked_state_len)


# ----------------------------------------------------------------- decay ----
def hla2_decay_forward(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, gamma: float,
                       O: torch.Tensor | None = None, normalized: bool = False,
                       workspace: torch.Tensor | None = None, state_out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Decayed masked forward, o_t = sum_{i<=j<=t} gamma^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j.
    Shapes and dtypes as for hla2_forward; ``state_out`` [B*H, d*d + d*dv + d]
    fp32 receives the final compact state S|P|p if given."""
    return _forward("hla2_decay_forward", Q, K, V, O, normalized, workspace, state_out, stream,
                    pform_record_len(*_dims(Q, V)), gamma=gamma)


def hla2_decay_step(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, gamma: float,
                    o: torch.Tensor | None = None, normalized: bool = False, stream=None) -> torch.Tensor:
    """One decayed decode step on the compact state [n, d*d + d*dv + d] (S|P|p, in place)."""
    return _step("hla2_decay_step", state, q, k, v, o, normalized, stream, pform_record_len, gamma=gamma)
