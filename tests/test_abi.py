"""The C-ABI library: builds, loads, exports every symbol include/hla2.h
declares, and rejects bad arguments on the host (no GPU work is issued)."""
import ctypes
import os
import re

import pytest

from higher_order_linear_gb300 import build as hbuild
from higher_order_linear_gb300 import hla2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hla2.h")


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return hla2.lib()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"HLA2_API\s+[\w\s\*]+?\b(hla2_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for want in ("hla2_forward", "hla2_forward_workspace", "hla2_step", "hla2_chunk_summaries", "hla2_scan",
                 "hla2_last_error_detail", "hla2_device_status"):
        assert want in syms


def test_every_declared_symbol_is_exported(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_workspace_query(L):
    R = lambda d, dv: d * d + 2 * d * dv + 2 * d
    # one head, T=64: one segment -> summary + prefix + total records and the
    # two decay factors of the segment, each rounded to 256 bytes
    ws = hla2.hla2_forward_workspace(1, 1, 64, 16, 16, 0)
    up = lambda n: (n + 63) // 64 * 64
    assert ws == 4 * (2 * up(R(16, 16)) + up(R(16, 16)) + up(2))
    big = hla2.hla2_forward_workspace(1, 16, 65536, 128, 128, 1)
    assert big > 0 and big % 256 == 0
    assert hla2.hla2_forward_workspace(1, 1, 64, 200, 16, 0) == 0   # unsupported d
    assert hla2.hla2_forward_workspace(1, 1, 0, 16, 16, 0) == 0     # empty
    assert hla2.hla2_forward_workspace(1, 1, 64, 16, 16, 7) == 0    # bad dtype


def _fake(addr=4096):
    return ctypes.c_void_p(addr)


def test_forward_rejects_bad_arguments(L):
    p = _fake()
    ws = hla2.hla2_forward_workspace(1, 1, 64, 16, 16, 0)
    assert L.hla2_forward(None, p, p, p, 1, 1, 64, 16, 16, 0, 0, p, ws, None, None) == hla2.HLA2_ERR_INVALID
    assert "null" in hla2.hla2_last_error_detail()
    assert L.hla2_forward(_fake(4097), p, p, p, 1, 1, 64, 16, 16, 0, 0, p, ws, None, None) == hla2.HLA2_ERR_INVALID
    assert "aligned" in hla2.hla2_last_error_detail()
    assert L.hla2_forward(p, p, p, p, 1, 1, 0, 16, 16, 0, 0, p, ws, None, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_forward(p, p, p, p, 1, 1, 64, 129, 16, 0, 0, p, ws, None, None) == hla2.HLA2_ERR_UNSUPPORTED
    assert L.hla2_forward(p, p, p, p, 1, 1, 64, 16, 16, 0, 3, p, ws, None, None) == hla2.HLA2_ERR_UNSUPPORTED
    assert L.hla2_forward(p, p, p, p, 1, 1, 64, 16, 16, 0, 0, p, ws - 1, None, None) == hla2.HLA2_ERR_WORKSPACE
    assert L.hla2_forward(p, p, p, p, 1, 1, 64, 16, 16, 0, 0, None, ws, None, None) == hla2.HLA2_ERR_WORKSPACE
    assert L.hla2_forward(p, p, p, p, 300, 300, 64, 16, 16, 0, 0, p, 1 << 40, None, None) == hla2.HLA2_ERR_UNSUPPORTED


def test_step_rejects_bad_arguments(L):
    p = _fake()
    assert L.hla2_step(None, p, p, p, p, 4, 16, 16, 0, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_step(p, p, p, p, p, 0, 16, 16, 0, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_step(p, p, p, p, p, 4, 12, 16, 0, None) == hla2.HLA2_ERR_UNSUPPORTED
    assert L.hla2_step(p, p, p, p, p, 4, 16, 256, 0, None) == hla2.HLA2_ERR_UNSUPPORTED
    assert L.hla2_step(p, _fake(4100), p, p, p, 4, 16, 16, 0, None) == hla2.HLA2_ERR_INVALID


def test_summaries_and_scan_reject_bad_arguments(L):
    p = _fake()
    assert L.hla2_chunk_summaries(p, p, p, p, 1, 1, 64, 16, 16, 0, 0, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_chunk_summaries(p, p, p, None, 1, 1, 64, 16, 16, 16, 0, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_scan(p, p, 1, 1, 4, 16, 16, None) == hla2.HLA2_ERR_INVALID  # overlap
    assert L.hla2_scan(p, _fake(1 << 30), 1, 1, 0, 16, 16, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_scan(p, _fake(1 << 30), 1, 1, 4, 130, 16, None) == hla2.HLA2_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(hla2, "_lib", None)
    monkeypatch.setattr(hla2, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        hla2.lib()


def _plan_restated(BH, T, sms):
    """The plan search restated from its description in include/hla2.h and
    hla2_api.cu: runs of `seglen` 128-token chunks (the last may be shorter),
    full runs dispatched first, each CTA costing its chunks + 2 on the first
    free of `sms` SMs; the run length minimises twice the makespan + nseg."""
    import heapq
    nchunk = (T + 127) // 128
    best = None
    for ln in range(max(1, (nchunk + 4095) // 4096), nchunk + 1):
        ns = (nchunk + ln - 1) // ln
        tail = nchunk - (ns - 1) * ln
        short = ns > 1 and tail < ln
        full = BH * (ns - 1) if short else BH * ns
        q, r = divmod(full, sms)
        span = (q + 1 if r else q) * (ln + 2)
        if short:
            if BH > 20000:
                span += -(-BH // sms) * (tail + 2)
            else:
                load = [(q + 1) * (ln + 2) if i < r else q * (ln + 2) for i in range(sms)]
                heapq.heapify(load)
                for _ in range(BH):
                    t = heapq.heappop(load) + tail + 2
                    heapq.heappush(load, t)
                    span = max(span, t)
        cost2 = 2 * span + ns
        if best is None or cost2 < best[0]:
            best = (cost2, ns, ln)
    return best[1], best[2]


PLAN_CASES = [(1, 16, 65536, 128), (4, 16, 4096, 64), (2, 8, 2048, 64), (1, 1, 65536, 128),
              (3, 1, 5000, 64), (1, 40, 200, 32), (1, 128, 16384, 128)]


@pytest.mark.parametrize("sms", [152, 148, 132, 76, 1])
@pytest.mark.parametrize("B,H,T,d", PLAN_CASES)
def test_plan_follows_the_sm_count(L, B, H, T, d, sms):
    """hla2_forward_plan with a faked SM count gives the plan the search
    describes for that count (the forward plans with the device's count)."""
    nseg, seglen, used = hla2.hla2_forward_plan(B, H, T, sm_count=sms)
    assert used == sms
    assert (nseg, seglen) == _plan_restated(B * H, T, sms)
    assert ((T + 127) // 128 + seglen - 1) // seglen == nseg


@pytest.mark.parametrize("B,H,T,d", PLAN_CASES)
def test_bench_plan_matches_workspace(L, B, H, T, d):
    """bench.py reports the plan it reads from the library; the workspace size
    (summaries, prefixes, totals, decay factors) pins that plan to the one the
    forward uses on the same device (152 SMs when none is visible)."""
    import bench
    nseg, seglen = bench.segments_per_head(B, H, T)
    assert (nseg, seglen) == hla2.hla2_forward_plan(B, H, T)[:2]
    R = d * d + 2 * d * d + 2 * d
    up = lambda n: (n + 63) // 64 * 64
    BH = B * H
    expect = 4 * (2 * up(BH * nseg * R) + up(BH * R) + up(2 * nseg))
    assert hla2.hla2_forward_workspace(B, H, T, d, d, hla2.HLA2_DTYPE_BF16) == expect


def test_plan_without_device_assumes_gb300(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is visible: the plan uses its SM count")
    assert hla2.hla2_forward_plan(1, 16, 65536)[2] == 152
    assert hla2.hla2_forward_plan(1, 16, 65536) == hla2.hla2_forward_plan(1, 16, 65536, sm_count=152)


def test_plan_rejects_bad_arguments(L):
    n = ctypes.c_int(0)
    assert L.hla2_forward_plan(0, 1, 64, 0, ctypes.byref(n), ctypes.byref(n), None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_forward_plan(1, 1, 64, 0, None, ctypes.byref(n), None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_forward_plan(300, 300, 64, 0, ctypes.byref(n), ctypes.byref(n), None) == hla2.HLA2_ERR_UNSUPPORTED


def test_host_forward_workspace_and_checks(L):
    """The host-buffer forward's device buffer holds two slots (a group's
    Q, K, V and O) and one forward workspace; its argument checks run on the
    host before any CUDA call."""
    up = lambda n: (n + 255) // 256 * 256
    B, H, T, d, dv, G = 1, 16, 4096, 64, 64, 3
    bf = hla2.HLA2_DTYPE_BF16
    slot = 2 * up(G * T * d * 2) + up(G * T * dv * 2) + up(G * T * dv * 4)
    last = B * H - (B * H + G - 1) // G * G + G  # heads in the last group
    ws = max(hla2.hla2_forward_workspace(1, G, T, d, dv, bf), hla2.hla2_forward_workspace(1, last, T, d, dv, bf))
    assert hla2.hla2_forward_host_workspace(B, H, T, d, dv, bf, G) == 2 * slot + up(ws)
    assert hla2.hla2_forward_host_workspace(B, H, T, d, dv, bf, 0) == hla2.hla2_forward_host_workspace(B, H, T, d, dv, bf, 2)
    assert hla2.hla2_forward_host_workspace(B, H, T, d, dv, bf, -1) == 0
    assert hla2.hla2_forward_host_workspace(B, H, T, 200, dv, bf, 0) == 0
    p = _fake()
    need = hla2.hla2_forward_host_workspace(B, H, T, d, dv, bf, G)
    dev = _fake(1 << 20)
    assert L.hla2_forward_host(None, p, p, p, B, H, T, d, dv, 0, bf, G, dev, need, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_forward_host(p, p, p, p, B, H, T, d, dv, 0, bf, -1, dev, need, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_forward_host(p, p, p, p, B, H, T, d, dv, 0, bf, G, dev, need - 1, None) == hla2.HLA2_ERR_WORKSPACE
    assert L.hla2_forward_host(p, p, p, p, B, H, T, d, dv, 0, bf, G, None, need, None) == hla2.HLA2_ERR_WORKSPACE
    assert L.hla2_forward_host(p, p, p, p, B, H, T, d, dv, 0, bf, G, _fake((1 << 20) + 16), need, None) == \
        hla2.HLA2_ERR_INVALID
    assert "aligned" in hla2.hla2_last_error_detail()
    assert L.hla2_forward_host(p, p, p, p, B, H, T, 200, dv, 0, bf, G, dev, need, None) == hla2.HLA2_ERR_UNSUPPORTED


def test_selftest_runout_rejects_bad_arguments(L):
    """The wait run-out self-test checks its arguments before any CUDA call."""
    assert L.hla2_selftest_wait_runout(None, 1000, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_selftest_wait_runout(_fake(4098), 1000, None) == hla2.HLA2_ERR_INVALID  # misaligned
    assert L.hla2_selftest_wait_runout(_fake(), 0, None) == hla2.HLA2_ERR_INVALID
    assert L.hla2_selftest_wait_runout(_fake(), 2000001, None) == hla2.HLA2_ERR_INVALID
    assert "wait_us" in hla2.hla2_last_error_detail()
