"""Guard regions around every buffer the library writes (a stand-in for a
memory sanitizer, which this pool does not offer): each output, state,
workspace and device staging buffer is carved out of a larger allocation
whose margins hold a byte pattern, and after the call every margin byte must
still hold it.  Inputs get margins too and must come back unchanged.

The forwards cover ragged sequence lengths (T = 1, 127, 129, 5000: one
token, one short of a chunk, one past a chunk, many chunks with a ragged
tail), d = dv in {64, 128}, both variants and all four operators, so the
tensor-core walks' clipped bulk stores of the last partial chunk and the
CUDA-core walks both run.  O is dense, so the margin after O is the space
past token T of the last head; inside O, a write past T of head h would land
on head h + 1, whose own outputs the parity tests check element by element.
"""
import dataclasses

import numpy as np
import pytest
import torch

from higher_order_linear_gb300 import hla2, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PATTERN = 0xA5
MARGIN = 64 * 1024  # bytes on each side (a multiple of 16: views stay aligned)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


class Guarded:
    """A tensor of `shape` inside an allocation with PATTERN-filled margins."""

    def __init__(self, shape, dtype, device=DEV, init=None, pin=False):
        esz = torch.empty((), dtype=dtype).element_size()
        self.m = MARGIN // esz
        self.n = int(np.prod(shape)) if len(shape) else 1
        kw = dict(dtype=dtype)
        if device == "cpu":
            self.buf = torch.empty(self.n + 2 * self.m, pin_memory=pin, **kw)
        else:
            self.buf = torch.empty(self.n + 2 * self.m, device=device, **kw)
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[self.m:self.m + self.n].view(shape)
        if init is not None:
            self.t.copy_(init)
        self.snapshot = self.t.clone() if init is not None else None

    def margins_intact(self) -> bool:
        torch.cuda.synchronize()
        b = self.buf.view(torch.uint8)
        esz = self.buf.element_size()
        lo, hi = b[:self.m * esz], b[(self.m + self.n) * esz:]
        return bool((lo == PATTERN).all()) and bool((hi == PATTERN).all())

    def unchanged(self) -> bool:
        torch.cuda.synchronize()
        return self.snapshot is not None and torch.equal(self.t, self.snapshot)


def _inputs(T, d, normalized, H=3):
    """The bf16 recipe of the d = 64 workloads (normal, or nonnegative q, k
    for the normalised variant) at head size d = dv."""
    w = dataclasses.replace(W.WORKLOADS[2] if normalized else W.WORKLOADS[1], d=d, dv=d)
    return W.make_inputs(w, B=1, H=H, T=T)


def _state_len(op, d, dv):
    return {"hla2": hla2.record_len, "ahla": hla2.ahla_state_len, "unmasked": hla2.unmasked_state_len,
            "decay": hla2.pform_record_len}[op](d, dv)


def _forward(op, q, k, v, O, normalized, ws, state_out, gamma):
    if op == "hla2":
        return hla2.hla2_forward(q, k, v, O, normalized=normalized, workspace=ws, state_out=state_out)
    if op == "ahla":
        return hla2.hla2_ahla_forward(q, k, v, O, normalized=normalized, workspace=ws, state_out=state_out)
    if op == "unmasked":
        return hla2.hla2_unmasked_forward(q, k, v, O, normalized=normalized, workspace=ws, state_out=state_out)
    return hla2.hla2_decay_forward(q, k, v, gamma, O, normalized=normalized, workspace=ws, state_out=state_out)


@pytest.mark.parametrize("op,gamma", [("hla2", None), ("ahla", None), ("unmasked", None), ("decay", 0.95),
                                      ("decay", 0.5)])
@pytest.mark.parametrize("normalized", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 127, 129, 5000])
def test_forward_writes_stay_inside(op, gamma, normalized, d, T):
    q, k, v = _inputs(T, d, normalized)
    B, H = q.shape[:2]
    dv = v.shape[-1]
    gq, gk, gv = (Guarded(x.shape, x.dtype, init=x.to(DEV)) for x in (q, k, v))
    gO = Guarded((B, H, T, dv), torch.float32)
    need = hla2.hla2_forward_workspace(B, H, T, d, dv, hla2.HLA2_DTYPE_BF16)
    gws = Guarded((need,), torch.uint8)
    for with_state in (False, True):
        gst = Guarded((B * H, _state_len(op, d, dv)), torch.float32) if with_state else None
        _forward(op, gq.t, gk.t, gv.t, gO.t, normalized, gws.t, gst.t if gst else None, gamma)
        assert hla2.hla2_device_status() == 0
        assert gO.margins_intact(), "O margin written"
        assert gws.margins_intact(), "workspace margin written"
        if gst:
            assert gst.margins_intact(), "state_out margin written"
            assert torch.isfinite(gst.t).all()
        assert gq.unchanged() and gk.unchanged() and gv.unchanged(), "an input was written"
        assert gq.margins_intact() and gk.margins_intact() and gv.margins_intact()
        assert torch.isfinite(gO.t).all()


@pytest.mark.parametrize("entry", ["hla2_step", "hla2_step_pform", "hla2_ahla_step", "hla2_unmasked_step",
                                   "hla2_decay_step"])
@pytest.mark.parametrize("d", [64, 128])
def test_step_writes_stay_inside(entry, d):
    n, dv = 5, d
    lens = {"hla2_step": hla2.record_len, "hla2_step_pform": hla2.pform_record_len,
            "hla2_ahla_step": hla2.ahla_state_len, "hla2_unmasked_step": hla2.unmasked_state_len,
            "hla2_decay_step": hla2.pform_record_len}
    gst = Guarded((n, lens[entry](d, dv)), torch.float32, init=torch.zeros(n, lens[entry](d, dv)))
    go = Guarded((n, dv), torch.float32)
    wd = W.DecodeWorkload("canary", n, d, dv, 0, 3, seed=21)
    fn = getattr(hla2, entry)
    for qt, kt, vt in W.decode_tokens(wd):
        gq, gk, gv = (Guarded(x.shape, torch.float32, init=x.to(DEV)) for x in (qt, kt, vt))
        if entry == "hla2_decay_step":
            fn(gst.t, gq.t, gk.t, gv.t, 0.9, o=go.t)
        else:
            fn(gst.t, gq.t, gk.t, gv.t, o=go.t)
        assert hla2.hla2_device_status() == 0
        assert gst.margins_intact() and go.margins_intact()
        assert gq.unchanged() and gk.unchanged() and gv.unchanged()
        assert gq.margins_intact() and gk.margins_intact() and gv.margins_intact()
        assert torch.isfinite(go.t).all()


@pytest.mark.parametrize("T", [127, 5000])
def test_host_forward_writes_stay_inside(T):
    """hla2_forward_host: the pinned host O and the device staging buffer."""
    q, k, v = _inputs(T, 64, False, H=5)
    B, H, _, d = q.shape
    dv = v.shape[-1]
    hq, hk, hv = (Guarded(x.shape, x.dtype, device="cpu", init=x, pin=True) for x in (q, k, v))
    hO = Guarded((B, H, T, dv), torch.float32, device="cpu", pin=True)
    need = hla2.hla2_forward_host_workspace(B, H, T, d, dv, hla2.HLA2_DTYPE_BF16, 2)
    gdev = Guarded((need,), torch.uint8)
    hla2.hla2_forward_host(hq.t, hk.t, hv.t, hO.t, heads_per_group=2, dev=gdev.t)
    torch.cuda.synchronize()
    assert hla2.hla2_device_status() == 0
    assert hO.margins_intact() and gdev.margins_intact()
    assert hq.unchanged() and hk.unchanged() and hv.unchanged()
    assert torch.isfinite(hO.t).all()


@pytest.mark.parametrize("T,L", [(129, 64), (1000, 100)])
def test_chunk_summaries_and_scan_writes_stay_inside(T, L):
    q, k, v = _inputs(T, 64, False, H=2)
    B, H, _, d = q.shape
    dv = v.shape[-1]
    N = (T + L - 1) // L
    R = hla2.record_len(d, dv)
    gq, gk, gv = (Guarded(x.shape, x.dtype, init=x.to(DEV)) for x in (q, k, v))
    gs = Guarded((B, H, N, R), torch.float32)
    gp = Guarded((B, H, N, R), torch.float32)
    hla2.hla2_chunk_summaries(gq.t, gk.t, gv.t, L, summ=gs.t)
    hla2.hla2_scan(gs.t, d, dv, prefix=gp.t)
    assert hla2.hla2_device_status() == 0
    assert gs.margins_intact() and gp.margins_intact()
    assert gq.unchanged() and gk.unchanged() and gv.unchanged()
    assert torch.isfinite(gp.t).all()
