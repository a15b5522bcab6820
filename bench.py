#!/usr/bin/env python
"""Benchmark of masked second-order HLA on one GB300 (or N replicas).

Headline: forward tokens/s (B*H*T per second) on the long-context workload
B=1 H=16 T=65536 d=dv=128, bf16 inputs, fp32 outputs, through hla2_forward.
A "step" is one hla2_forward over that batch: segment summaries, exclusive
scan, segment outputs.  Inputs (1.3 GB read + written per step) exceed the
129 MB L2, so no flush is needed between steps.

Also reported on the same line:
  roofline      dominant kernel (segment outputs) against measured HBM peak;
  e2e           the same metric through the public API with pinned host
                buffers, host->device inputs and device->host outputs timed;
  decode        hla2_step tokens/s on n=4096 heads, d=dv=128 (fp32 state),
                with its own HBM roofline;
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample.
`--impl reference` times the oracle alone as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload
(independent heads, no collective on the data path); value = all ranks'
tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked HLA-2 fwd tokens/s (B·H·T/s) at 1 GB300; % tensor/HBM roofline"
UNIT = "tokens/s"
FWD_WORKLOAD = 3          # B1 H16 T65536 d=dv=128 bf16
BYTES_PER_TOKEN_FWD = None  # set from the workload: 2*(2d+dv) + 4*dv
# ncu DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum),
# valid only for the kernel source it was taken on, keyed by (kernel, workload).
# Both were captured at full size with one-pass metrics (profiles/*.md give
# the commands and the raw figures):
#  - tc_out_kernel<128> (the output walk), B1 H16 T65536: 826.4 + 489.2 MB;
#  - decode step_kernel, 4096 heads: 815.9 + 752.5 MB.
# Writes still in L2 when a kernel ends are not counted, so the write side
# sits a little below the algorithmic bytes.
NCU_TRAFFIC = {
    ("tcgen05", "hla2-fwd-B1H16T65536-d128-bf16"): 826415968 + 489178976,  # tc_out_kernel<128>
    ("step", "hla2-step-n4096-d128-fp32-prefill1024-steps512"): 815852544 + 752451328,
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU seconds for the oracle sample")
    p.add_argument("--no-forward", action="store_true", help="skip the forward (profiling the decode step alone)")
    p.add_argument("--T", type=int, default=None, help="override T (profiling a smaller case; not a bench line)")
    p.add_argument("--H", type=int, default=None, help="override H (profiling a smaller case; not a bench line)")
    p.add_argument("--no-ahla", action="store_true", help="skip the AHLA forward and decode lines")
    p.add_argument("--no-small", action="store_true",
                   help="skip the B2 H8 T2048 d64 forward timed eagerly and as a CUDA graph")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the unmasked and decayed forward and decode lines")
    p.add_argument("--decode-n", type=int, default=None,
                   help="override the number of decode heads (profiling a smaller case; not a bench line)")
    p.add_argument("--no-normalized", action="store_true",
                   help="skip the ratio-normalised B4 H16 T4096 d64 forward line")
    p.add_argument("--no-chunk-level", action="store_true",
                   help="skip timing hla2_chunk_summaries (L = 64) and hla2_scan on the headline inputs")
    p.add_argument("--workload", type=int, default=FWD_WORKLOAD,
                   help="forward workload id (0-3, see workloads.py); the bench line is workload 3")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        import torch
        fd, self.path = tempfile.mkstemp(prefix="hla2_clocks_", suffix=".csv")
        os.close(fd)
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100", *sel]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # nvidia-smi samples every 100 ms; keep those taken while the timed work ran
        n = len(rows)
        span = max(1e-6, time.time() - self.t0)
        idx = [i for i in range(n) if t_begin - self.t0 <= (i + 0.5) * span / n <= t_end - self.t0 + 0.1]
        sel = [rows[i] for i in idx] or rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in sel if num(r[1]) is not None]
        mx = [num(r[2]) for r in sel if num(r[2]) is not None]
        pw = [num(r[3]) for r in sel if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(sel), "reasons": sorted(reasons)}


# ------------------------------------------------------------- oracle leg --
def oracle_sample(w, seconds: float):
    """Time the fp64 oracle on all heads of the workload, first T_s tokens,
    T_s sized for about `seconds` of CPU time.  Returns (tokens/s, cores, sample)."""
    import oracle
    from higher_order_linear_gb300 import workloads as W
    cores = os.cpu_count() or 1
    threads = min(cores, w.BH)
    oracle.build()

    def run(T):
        q, k, v = W.make_inputs(w, T=T)
        Q, K, V = (x.double().numpy() for x in (q, k, v))
        t0 = time.perf_counter()
        oracle.serial(Q, K, V, normalized=w.normalized, nthreads=threads)
        return time.perf_counter() - t0

    T_cal = min(w.T, 512)
    t_cal = run(T_cal)
    T_s = int(min(w.T, max(T_cal, T_cal * seconds / max(t_cal, 1e-6))))
    t = run(T_s) if T_s != T_cal else t_cal
    return w.BH * T_s / t, threads, f"all {w.BH} heads x first {T_s} of {w.T} tokens (same recipe), {t:.1f} s"


# ----------------------------------------------------------------- config --
def fwd_config(w, plan_segments=None, l2_note=None):
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "input_dtype": w.dtype,
            "output_dtype": "fp32", "normalized": w.normalized,
            "segments_per_head": plan_segments[0] if plan_segments else None,
            "chunks_per_segment": plan_segments[1] if plan_segments else None,
            "l2": l2_note or "inputs exceed L2 (1.34 GB moved per step vs 129 MB L2); no flush",
            "parallelism": "replicas (heads independent, no collective)"}


def alg_flops(w, L=64):
    """Algorithmic flops per token-head of the chunked forward (fixed count,
    chunk L = 64): 2 [2 L d + L^2 + 2 d^2 + 2 L dv + 3 d dv]."""
    return 2 * (2 * L * w.d + L * L + 2 * w.d * w.d + 2 * L * w.dv + 3 * w.d * w.dv)


def segments_per_head(B, H, T):
    """The library's segment plan for the current device (its SM count
    queried by the library): (segments per head, chunks per segment)."""
    from higher_order_linear_gb300 import hla2
    nseg, seglen, _ = hla2.hla2_forward_plan(B, H, T)
    return nseg, seglen


def reference_arm(args):
    from higher_order_linear_gb300 import workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.WORKLOADS[FWD_WORKLOAD]
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    threads = min(cores, w.BH)
    # each step: all heads, first T_s tokens, sized for ~2 s of CPU work
    T_cal = 256
    q, k, v = W.make_inputs(w, T=T_cal)
    t0 = time.perf_counter()
    oracle.serial(q.double().numpy(), k.double().numpy(), v.double().numpy(), nthreads=threads)
    t_cal = time.perf_counter() - t0
    T_s = int(min(w.T, max(T_cal, T_cal * 2.0 / max(t_cal, 1e-6))))
    q, k, v = W.make_inputs(w, T=T_s)
    Q, K, V = (x.double().numpy() for x in (q, k, v))
    for _ in range(args.warmup):
        oracle.serial(Q, K, V, nthreads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.serial(Q, K, V, nthreads=threads)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = w.BH * T_s * args.steps / tot
    sample = f"each step: all {w.BH} heads x first {T_s} of {w.T} tokens (same recipe), fp64 serial recurrence"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": fwd_config(w, segments_per_head(w.B, w.H, w.T)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours --
def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch
    import torch.distributed as dist
    from higher_order_linear_gb300 import build as hbuild, hla2, replicas, workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        raise SystemExit(f"WORLD_SIZE={world} but --gpus {args.gpus}")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    hbuild.build()
    L = hla2.lib()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return replicas.max_over_ranks(x, dev)

    peaks = load_peaks()
    w = W.WORKLOADS[args.workload]
    if args.T or args.H:
        w = dataclasses.replace(w, T=args.T or w.T, H=args.H or w.H, name=w.name + f"-override-H{args.H or w.H}-T{args.T or w.T}")
    tokens = w.BH * w.T
    esz = 2 if w.dtype == "bf16" else 4
    bytes_per_token = esz * (2 * w.d + w.dv) + 4 * w.dv  # read Q,K,V once, write O fp32 once
    q, k, v = W.make_inputs_on(w, dev, seed=w.seed + 1000 * rank)
    O = torch.empty(w.B, w.H, w.T, w.dv, device=dev, dtype=torch.float32)
    dcode = hla2.HLA2_DTYPE_BF16 if w.dtype == "bf16" else hla2.HLA2_DTYPE_F32
    need = hla2.hla2_forward_workspace(w.B, w.H, w.T, w.d, w.dv, dcode)
    ws = torch.empty(need, device=dev, dtype=torch.uint8)
    path = "tcgen05" if L.hla2_forward_path(w.d, w.dv, dcode, int(w.normalized), 0) == 1 else "cuda-core"

    clocks = ClockSampler(local)
    clocks.start()
    fwd_steps = 0 if args.no_forward else args.steps
    for _ in range(0 if args.no_forward else args.warmup):
        hla2.hla2_forward(q, k, v, O, normalized=w.normalized, workspace=ws)
    barrier()
    stream = torch.cuda.current_stream()
    # Workloads whose step moves less than 4x the 129 MB L2 flush it (outside
    # the timed events) before every step; larger ones stream from HBM anyway.
    step_bytes = bytes_per_token * tokens
    flush = step_bytes < 4 * 129e6
    l2_note = ("L2 flushed before every step (256 MB write outside the timed events)" if flush else
               f"inputs exceed L2 ({step_bytes / 1e9:.2f} GB moved per step vs 129 MB L2); no flush")
    scratch = torch.empty(64 << 20, device=dev, dtype=torch.float32)  # 256 MB: flushes L2 where asked

    def timed(call, n, flush_each):
        """Mean ms of `call` over n steps, CUDA events on the launching stream;
        with flush_each, L2 is flushed before every step outside the events."""
        if flush_each:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for ea, eb in evs:
                scratch.zero_()
                ea.record(stream)
                call()
                eb.record(stream)
            barrier()
            return sum(ea.elapsed_time(eb) for ea, eb in evs) / n
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / n

    fwd = lambda: hla2.hla2_forward(q, k, v, O, normalized=w.normalized, workspace=ws)
    # The headline is timed bare (no per-phase events recorded); the library's
    # launch counter, which costs nothing on the GPU, counts its launches.
    hla2.hla2_profile_enable(False)
    hla2.hla2_profile_read()  # resets the launch counter
    t_begin = time.time()
    ms_step = timed(fwd, fwd_steps, flush) if fwd_steps else 0.0
    t_end = time.time()
    _, _, launches = hla2.hla2_profile_read()
    ms_step_max = max_over_ranks(ms_step)
    status = hla2.hla2_device_status()
    if status != 0:
        raise SystemExit(f"device status {status}: {hla2.hla2_last_error_detail()}")
    value = replicas.job_throughput(tokens, world, ms_step_max) if fwd_steps else 0.0

    def phase_split(call, n, flush_each):
        """A separate instrumented run: the library records CUDA events on the
        launching stream around each phase (summaries, scan, outputs) of n
        forwards.  Returns (per-phase ms per forward, ms per instrumented step)."""
        hla2.hla2_profile_read()
        hla2.hla2_profile_enable(True)
        ms_instr = timed(call, n, flush_each)
        hla2.hla2_profile_enable(False)
        ph, nf, _ = hla2.hla2_profile_read()
        return [x / max(nf, 1) for x in ph], ms_instr

    n_prof = max(1, min(args.steps, 20))
    phase, ms_instr = phase_split(fwd, n_prof, flush) if fwd_steps else ([0.0, 0.0, 0.0], 0.0)

    # dominant kernel: segment outputs (phase 2)
    out_ms = phase[2]
    achieved = bytes_per_token * tokens / (out_ms / 1e3) / 1e9 if out_ms > 0 else 0.0
    traffic = NCU_TRAFFIC.get((path, w.name))
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": f"segment outputs ({path})", "ms_per_launch": out_ms,
                "phase_ms_per_step": {"summaries": phase[0], "scan": phase[1], "outputs": out_ms},
                "phase_source": f"separate instrumented run of {n_prof} forwards "
                                f"({ms_instr:.4f} ms per step with the per-phase events)",
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS hbm_gbs)" if peaks["source"] == "measured"
                else "fallback 6.8 TB/s",
                "step_frac": bytes_per_token * tokens / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"] if fwd_steps else 0.0,
                "tensor_frac_of_bf16_burst": (alg_flops(w) * tokens / (ms_step / 1e3) / 1e12) / peaks["bf16_tflops"]
                if fwd_steps else 0.0}

    # ---- the same forward handing over each head's final state (prefill ->
    # decode), timed like the headline ----
    with_state = None
    if fwd_steps:
        st = torch.empty(w.B * w.H, hla2.record_len(w.d, w.dv), device=dev, dtype=torch.float32)
        sfwd = lambda: hla2.hla2_forward(q, k, v, O, normalized=w.normalized, workspace=ws, state_out=st)
        for _ in range(args.warmup):
            sfwd()
        barrier()
        n_s = max(1, min(args.steps, 50))
        ms_s = max_over_ranks(timed(sfwd, n_s, flush))
        if hla2.hla2_device_status() != 0:
            raise SystemExit(f"device status after the forward with state_out: {hla2.hla2_last_error_detail()}")
        with_state = {"ms_per_step": ms_s, "steps": n_s, "value": replicas.job_throughput(tokens, world, ms_s),
                      "unit": UNIT, "vs_headline_ms": ms_s / ms_step_max if ms_step_max > 0 else None,
                      "path": "tcgen05" if L.hla2_forward_path(w.d, w.dv, dcode, int(w.normalized), 1) == 1
                      else "cuda-core"}
        del st

    # ---- the ratio-normalised workload (B4 H16 T4096 d=dv=64, q, k >= 0) ----
    normalized = None
    if not args.no_normalized and fwd_steps and args.workload == FWD_WORKLOAD and not (args.T or args.H):
        wn = W.WORKLOADS[2]
        nq, nk, nv = W.make_inputs_on(wn, dev, seed=wn.seed + 1000 * rank)
        nO = torch.empty(wn.B, wn.H, wn.T, wn.dv, device=dev, dtype=torch.float32)
        ncode = hla2.HLA2_DTYPE_BF16
        nws = torch.empty(max(hla2.hla2_forward_workspace(wn.B, wn.H, wn.T, wn.d, wn.dv, ncode), 16),
                          device=dev, dtype=torch.uint8)
        npath = "tcgen05" if L.hla2_forward_path(wn.d, wn.dv, ncode, 1, 0) == 1 else "cuda-core"
        nfwd = lambda: hla2.hla2_forward(nq, nk, nv, nO, normalized=True, workspace=nws)
        for _ in range(args.warmup):
            nfwd()
        barrier()
        ntok = wn.B * wn.H * wn.T
        nbytes_tok = 2 * (2 * wn.d + wn.dv) + 4 * wn.dv
        nflush = nbytes_tok * ntok < 4 * 129e6
        n_n = max(1, min(args.steps, 50))
        ms_n = max_over_ranks(timed(nfwd, n_n, nflush))
        nphase, nms_instr = phase_split(nfwd, max(1, min(n_n, 20)), nflush)
        if hla2.hla2_device_status() != 0:
            raise SystemExit(f"device status after the normalised forward: {hla2.hla2_last_error_detail()}")
        n_ach = nbytes_tok * ntok / (nphase[2] / 1e3) / 1e9 if nphase[2] > 0 else 0.0
        normalized = {
            "metric": "ratio-normalised HLA-2 fwd tokens/s (B·H·T/s)", "workload": wn.name,
            "value": replicas.job_throughput(ntok, world, ms_n), "unit": UNIT, "ms_per_step": ms_n, "steps": n_n,
            "path": npath,
            "l2": (f"L2 flushed before every step (256 MB write outside the timed events); "
                   f"{nbytes_tok * ntok / 1e6:.1f} MB moved per step vs 129 MB L2") if nflush else "no flush",
            "roofline": {"bound": "hbm", "achieved": n_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": n_ach / peaks["hbm_gbs"], "traffic": None,
                         "kernel": f"segment outputs ({npath}, normalised)", "ms_per_launch": nphase[2],
                         "bytes_per_token_head": nbytes_tok,
                         "phase_ms_per_step": {"summaries": nphase[0], "scan": nphase[1], "outputs": nphase[2]},
                         "step_frac": nbytes_tok * ntok / (ms_n / 1e3) / 1e9 / peaks["hbm_gbs"]}}
        del nq, nk, nv, nO, nws

    # ---- the chunk-level calls of the boundary on the headline inputs:
    # hla2_chunk_summaries (L = 64: 1024 chunks per head) and hla2_scan ----
    chunk_level = None
    if not args.no_chunk_level and fwd_steps and args.workload == FWD_WORKLOAD and not (args.T or args.H):
        Lc = 64
        N = (w.T + Lc - 1) // Lc
        R = hla2.record_len(w.d, w.dv)
        summ = torch.empty(w.B, w.H, N, R, device=dev, dtype=torch.float32)
        pref = torch.empty_like(summ)
        cs = lambda: hla2.hla2_chunk_summaries(q, k, v, Lc, summ=summ)
        sc = lambda: hla2.hla2_scan(summ, w.d, w.dv, prefix=pref)
        cs()
        sc()
        barrier()
        n_c = max(1, min(args.steps, 3))
        ms_cs = max_over_ranks(timed(cs, n_c, False))
        ms_sc = max_over_ranks(timed(sc, n_c, False))
        if hla2.hla2_device_status() != 0:
            raise SystemExit(f"device status after the chunk-level calls: {hla2.hla2_last_error_detail()}")
        rec_bytes = w.BH * N * R * 4
        cs_bytes = esz * (2 * w.d + w.dv) * tokens + rec_bytes  # read Q, K, V; write the records
        sc_bytes = 2 * rec_bytes                                 # read the records; write the prefixes
        chunk_level = {
            "L": Lc, "chunks_per_head": N, "record_bytes": R * 4,
            "chunk_summaries": {"ms": ms_cs, "steps": n_c, "algorithmic_bytes": cs_bytes,
                                "roofline": {"bound": "hbm", "achieved": cs_bytes / (ms_cs / 1e3) / 1e9,
                                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                             "frac": cs_bytes / (ms_cs / 1e3) / 1e9 / peaks["hbm_gbs"]}},
            "scan": {"ms": ms_sc, "steps": n_c, "algorithmic_bytes": sc_bytes,
                     "roofline": {"bound": "hbm", "achieved": sc_bytes / (ms_sc / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": sc_bytes / (ms_sc / 1e3) / 1e9 / peaks["hbm_gbs"]}},
            "note": "records are S|C|m|G|h fp32 per chunk; both calls are bound by writing / reading them"}
        del summ, pref

    # ---- AHLA (asymmetric variant) forward on the same inputs ----
    ahla = None
    if not args.no_ahla and fwd_steps:
        apath = "tcgen05" if L.hla2_ahla_forward_path(w.d, w.dv, dcode, int(w.normalized), 0) == 1 else "cuda-core"
        for _ in range(args.warmup):
            hla2.hla2_ahla_forward(q, k, v, O, normalized=w.normalized, workspace=ws)
        barrier()
        n_a = max(1, min(args.steps, 50))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_a)]
        for ea, eb in evs:
            if flush:
                scratch.zero_()
            ea.record(stream)
            hla2.hla2_ahla_forward(q, k, v, O, normalized=w.normalized, workspace=ws)
            eb.record(stream)
        barrier()
        ms_a = max_over_ranks(sum(ea.elapsed_time(eb) for ea, eb in evs) / n_a)
        if hla2.hla2_device_status() != 0:
            raise SystemExit(f"device status after AHLA: {hla2.hla2_last_error_detail()}")
        ach_a = bytes_per_token * tokens / (ms_a / 1e3) / 1e9
        ahla = {"metric": "masked AHLA fwd tokens/s (B·H·T/s)", "value": replicas.job_throughput(tokens, world, ms_a),
                "unit": UNIT, "ms_per_step": ms_a, "steps": n_a, "path": apath,
                "roofline": {"bound": "hbm", "achieved": ach_a, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": ach_a / peaks["hbm_gbs"], "traffic": None,
                             "kernel": "whole AHLA forward step (summaries + scan + outputs)"}}

    # ---- the other operators on the same inputs: unmasked and decayed ----
    # (a few timed steps keep the run short)
    variants = None
    if not args.no_variants and fwd_steps:
        variants = {}
        gamma = 0.999
        for name, call in (("unmasked", lambda: hla2.hla2_unmasked_forward(q, k, v, O, normalized=w.normalized,
                                                                           workspace=ws)),
                           ("decay", lambda: hla2.hla2_decay_forward(q, k, v, gamma, O, normalized=w.normalized,
                                                                     workspace=ws))):
            call()
            barrier()
            n_v = 3
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(n_v):
                call()
            ev1.record(stream)
            barrier()
            ms_v = max_over_ranks(ev0.elapsed_time(ev1) / n_v)
            if hla2.hla2_device_status() != 0:
                raise SystemExit(f"device status after {name}: {hla2.hla2_last_error_detail()}")
            ach_v = bytes_per_token * tokens / (ms_v / 1e3) / 1e9
            if name == "unmasked":
                tc_v = L.hla2_unmasked_forward_path(w.d, w.dv, dcode, int(w.normalized), 0) == 1
            else:
                tc_v = L.hla2_decay_forward_path(w.d, w.dv, dcode, int(w.normalized), 0, gamma) == 1
            if tc_v:
                roof_v = {"bound": "hbm", "achieved": ach_v, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": ach_v / peaks["hbm_gbs"], "traffic": None,
                          "kernel": f"whole {name} forward step (summaries + scan + outputs)"}
            else:
                roof_v = {"bound": "alu", "hbm_frac": ach_v / peaks["hbm_gbs"],
                          "note": "fp32 CUDA-core walks; HBM fraction given for scale"}
            variants[name] = {"metric": f"{name} fwd tokens/s (B·H·T/s)", "value": replicas.job_throughput(tokens, world, ms_v),
                              "unit": UNIT, "ms_per_step": ms_v, "steps": n_v,
                              "path": "tcgen05" if tc_v else "cuda-core", "roofline": roof_v}
        variants["decay"]["gamma"] = gamma

    # ---- the latency-scale workload (B2 H8 T2048 d64): eager launches and a
    # CUDA graph of the same forwards, replayed ----
    small = None
    if not args.no_small and not args.no_forward and rank == 0:
        ws1 = W.WORKLOADS[1]
        sq, sk, sv = W.make_inputs_on(ws1, dev)
        sO = torch.empty(ws1.B, ws1.H, ws1.T, ws1.dv, device=dev, dtype=torch.float32)
        sws = torch.empty(max(hla2.hla2_forward_workspace(ws1.B, ws1.H, ws1.T, ws1.d, ws1.dv,
                                                          hla2.HLA2_DTYPE_BF16), 16), device=dev, dtype=torch.uint8)
        n_in = 20  # forwards per graph
        for _ in range(3):
            hla2.hla2_forward(sq, sk, sv, sO, workspace=sws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(100):
            hla2.hla2_forward(sq, sk, sv, sO, workspace=sws)
        e1.record()
        torch.cuda.synchronize()
        ms_eager = e0.elapsed_time(e1) / 100
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            hla2.hla2_forward(sq, sk, sv, sO, workspace=sws)  # first call outside the capture
            cs.synchronize()
            with torch.cuda.graph(g, stream=cs):
                for _ in range(n_in):
                    hla2.hla2_forward(sq, sk, sv, sO, workspace=sws)
        torch.cuda.synchronize()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(5):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_graph = e0.elapsed_time(e1) / (5 * n_in)
        if hla2.hla2_device_status() != 0:
            raise SystemExit(f"device status after the graph replays: {hla2.hla2_last_error_detail()}")
        ntok = ws1.B * ws1.H * ws1.T
        small = {"workload": ws1.name, "metric": "masked HLA-2 fwd tokens/s (B·H·T/s)",
                 "eager": {"value": ntok / (ms_eager / 1e3), "ms_per_forward": ms_eager, "forwards": 100},
                 "graph": {"value": ntok / (ms_graph / 1e3), "ms_per_forward": ms_graph,
                           "forwards": 5 * n_in, "forwards_per_graph": n_in},
                 "unit": UNIT, "inputs_in_l2": True,
                 "note": "inputs (12.6 MB) stay in L2 between forwards: a latency-scale case, not an HBM roofline"}
        del sq, sk, sv, sO, sws, g

    # ---- e2e through the C ABI with pinned host buffers: hla2_forward_host
    # copies Q, K, V in and O out itself, pipelined over groups of heads ----
    e2e = None
    if not args.no_e2e and not args.no_forward:
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hO = torch.empty(O.shape, dtype=torch.float32).pin_memory()
        n_e2e = max(2, min(args.steps, 10))
        del ws  # the host call has its own device buffer (two slots and a workspace)
        dcode_e = hla2.HLA2_DTYPE_BF16 if w.dtype == "bf16" else hla2.HLA2_DTYPE_F32
        hdev = torch.empty(hla2.hla2_forward_host_workspace(w.B, w.H, w.T, w.d, w.dv, dcode_e, 0),
                           dtype=torch.uint8, device=dev)
        for _ in range(2):
            hla2.hla2_forward_host(hq, hk, hv, hO, normalized=w.normalized, dev=hdev)
        barrier()
        e2 = torch.cuda.Event(enable_timing=True); e3 = torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n_e2e):
            hla2.hla2_forward_host(hq, hk, hv, hO, normalized=w.normalized, dev=hdev)
        e3.record(stream)
        barrier()
        ms_e2e = max_over_ranks(e2.elapsed_time(e3) / n_e2e)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h = hO.numel() * hO.element_size()
        e2e = {"value": world * tokens / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "steps": n_e2e,
               "api": "hla2_forward_host (copies in, forward and copy out pipelined over groups of heads)"}
        del hq, hk, hv, hO, hdev

    # ---- decode: hla2_step on n=4096 heads, d=dv=128 ----
    decode = None
    if not args.no_decode:
        wd = W.DECODE if args.decode_n is None else dataclasses.replace(
            W.DECODE, n=args.decode_n, name=W.DECODE.name + f"-override-n{args.decode_n}")
        R = W.state_floats(wd.d, wd.dv)
        state = torch.zeros(wd.n, R, device=dev)
        toks = list(W.decode_tokens(wd, device=dev, seed=wd.seed + 1000 * rank))
        for t in range(wd.prefill):
            hla2.hla2_step(state, *toks[t])
        barrier()
        o = torch.empty(wd.n, wd.dv, device=dev)
        e4 = torch.cuda.Event(enable_timing=True); e5 = torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        for t in range(wd.prefill, wd.prefill + wd.steps):
            hla2.hla2_step(state, *toks[t], o=o)
        e5.record(stream)
        barrier()
        ms_dec = max_over_ranks(e4.elapsed_time(e5) / wd.steps)
        bytes_head = 8 * R + 4 * (2 * wd.d + 2 * wd.dv)
        ach = wd.n * bytes_head / (ms_dec / 1e3) / 1e9
        decode = {"metric": "hla2_step tokens/s (heads*steps/s)", "workload": wd.name,
                  "value": world * wd.n / (ms_dec / 1e3), "unit": "tokens/s", "ms_per_step": ms_dec,
                  "steps": wd.steps, "prefill": wd.prefill,
                  "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": ach / peaks["hbm_gbs"], "traffic": NCU_TRAFFIC.get(("step", wd.name)),
                               "bytes_per_head_step": bytes_head}}
        # the same stream on the compact P-form state (S | P | p), converted from the prefilled state
        Rp = hla2.pform_record_len(wd.d, wd.dv)
        del state
        pstate = torch.zeros(wd.n, Rp, device=dev)
        for t in range(wd.prefill):
            hla2.hla2_step_pform(pstate, *toks[t])
        barrier()
        e6 = torch.cuda.Event(enable_timing=True); e7 = torch.cuda.Event(enable_timing=True)
        e6.record(stream)
        for t in range(wd.prefill, wd.prefill + wd.steps):
            hla2.hla2_step_pform(pstate, *toks[t], o=o)
        e7.record(stream)
        barrier()
        ms_pf = max_over_ranks(e6.elapsed_time(e7) / wd.steps)
        bytes_pf = 8 * Rp + 4 * (2 * wd.d + 2 * wd.dv)
        ach_pf = wd.n * bytes_pf / (ms_pf / 1e3) / 1e9
        decode["pform"] = {"metric": "hla2_step_pform tokens/s (heads*steps/s)", "value": world * wd.n / (ms_pf / 1e3),
                           "unit": "tokens/s", "ms_per_step": ms_pf,
                           "roofline": {"bound": "hbm", "achieved": ach_pf, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": ach_pf / peaks["hbm_gbs"], "bytes_per_head_step": bytes_pf}}
        if not args.no_ahla:
            # AHLA decode on the same token stream: state P | E | m | n per head
            Ra = hla2.ahla_state_len(wd.d, wd.dv)
            del pstate
            astate = torch.zeros(wd.n, Ra, device=dev)
            for t in range(wd.prefill):
                hla2.hla2_ahla_step(astate, *toks[t])
            barrier()
            e8 = torch.cuda.Event(enable_timing=True); e9 = torch.cuda.Event(enable_timing=True)
            e8.record(stream)
            for t in range(wd.prefill, wd.prefill + wd.steps):
                hla2.hla2_ahla_step(astate, *toks[t], o=o)
            e9.record(stream)
            barrier()
            ms_ah = max_over_ranks(e8.elapsed_time(e9) / wd.steps)
            bytes_ah = 8 * Ra + 4 * (2 * wd.d + 2 * wd.dv)
            ach_ah = wd.n * bytes_ah / (ms_ah / 1e3) / 1e9
            decode["ahla"] = {"metric": "hla2_ahla_step tokens/s (heads*steps/s)",
                              "value": world * wd.n / (ms_ah / 1e3), "unit": "tokens/s", "ms_per_step": ms_ah,
                              "roofline": {"bound": "hbm", "achieved": ach_ah, "peak": peaks["hbm_gbs"],
                                           "unit": "GB/s", "frac": ach_ah / peaks["hbm_gbs"],
                                           "bytes_per_head_step": bytes_ah}}
            pstate = astate
        if not args.no_variants:
            # unmasked (S | C | m) and decayed (S | P | p) decode steps on the same stream
            Rp = hla2.pform_record_len(wd.d, wd.dv)
            del pstate
            for name, step in (("unmasked", lambda st, t: hla2.hla2_unmasked_step(st, *t, o=o)),
                               ("decay", lambda st, t: hla2.hla2_decay_step(st, *t, 0.999, o=o))):
                vstate = torch.zeros(wd.n, Rp, device=dev)
                for t in range(64):  # the state's values do not change the work per step
                    step(vstate, toks[t])
                barrier()
                e10 = torch.cuda.Event(enable_timing=True); e11 = torch.cuda.Event(enable_timing=True)
                e10.record(stream)
                for t in range(wd.prefill, wd.prefill + wd.steps):
                    step(vstate, toks[t])
                e11.record(stream)
                barrier()
                ms_s = max_over_ranks(e10.elapsed_time(e11) / wd.steps)
                bytes_s = 8 * Rp + 4 * (2 * wd.d + 2 * wd.dv)
                ach_s = wd.n * bytes_s / (ms_s / 1e3) / 1e9
                decode[name] = {"metric": f"{name} decode tokens/s (heads*steps/s)",
                                "value": world * wd.n / (ms_s / 1e3), "unit": "tokens/s", "ms_per_step": ms_s,
                                "roofline": {"bound": "hbm", "achieved": ach_s, "peak": peaks["hbm_gbs"],
                                             "unit": "GB/s", "frac": ach_s / peaks["hbm_gbs"],
                                             "bytes_per_head_step": bytes_s}}
                del vstate
            pstate = None
        del toks, pstate
    clk = clocks.stop(t_begin, t_end)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, cores, sample = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if path == "tcgen05" else "f32", "data": "synthetic",
                "config": fwd_config(w, segments_per_head(w.B, w.H, w.T), l2_note), "path": path,
                "clocks": clk, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
                "cpu_baseline": cpu, "decode": decode, "ahla": ahla, "variants": variants, "small": small,
                "normalized": normalized, "chunk_level": chunk_level, "with_state_out": with_state}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
