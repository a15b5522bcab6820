"""Seeded synthetic inputs for masked second-order HLA.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can take their
inputs from it.  Every tensor is drawn on the CPU with a ``torch.Generator``
seeded per workload, in a fixed order (q, then k, then v), as fp32, scaled,
then cast to the workload's input type with round-to-nearest-even.

The five workloads are the ones the method is exercised on:

==  =====================================================================
0   B=1 H=1 T=64 d=dv=16, fp32, q,k,v ~ N(0,1)/sqrt(d), chunk 16, seed 0
1   B=2 H=8 T=2048 d=dv=64, bf16, q,k,v ~ N(0,1)/sqrt(d), chunk 64, seed 1
2   B=4 H=16 T=4096 d=dv=64, bf16, ratio-normalised, q,k ~ U(0,1)/sqrt(d),
    v ~ N(0,1), seed 2 (nonnegative q,k keep the denominator positive)
3   B=1 H=16 T=65536 d=dv=128, bf16, q,k,v ~ N(0,1)/sqrt(d), 1024 chunks
    of 64, seed 3
4   decode: 256 sequences x 16 heads (n=4096), d=dv=128, fp32 state;
    1024 prefill tokens then 512 single-token steps, N(0,1)/sqrt(d), seed 4
==  =====================================================================
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dv: int
    dtype: str            # "fp32" or "bf16": the input type
    normalized: bool
    chunk: int
    seed: int
    qk_dist: str = "normal"   # "normal": N(0,1)/sqrt(d); "uniform": U(0,1)/sqrt(d)
    v_dist: str = "normal"    # "normal": N(0,1)/sqrt(d); "unit": N(0,1)

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


WORKLOADS = {
    0: Workload("hla2-fwd-B1H1T64-d16-fp32", 1, 1, 64, 16, 16, "fp32", False, 16, 0),
    1: Workload("hla2-fwd-B2H8T2048-d64-bf16", 2, 8, 2048, 64, 64, "bf16", False, 64, 1),
    2: Workload("hla2-fwd-normalized-B4H16T4096-d64-bf16", 4, 16, 4096, 64, 64, "bf16", True, 64, 2,
                qk_dist="uniform", v_dist="unit"),
    3: Workload("hla2-fwd-B1H16T65536-d128-bf16", 1, 16, 65536, 128, 128, "bf16", False, 64, 3),
}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    n: int          # sequences x heads
    d: int
    dv: int
    prefill: int
    steps: int
    seed: int
    normalized: bool = False


DECODE = DecodeWorkload("hla2-step-n4096-d128-fp32-prefill1024-steps512", 4096, 128, 128, 1024, 512, 4)


def _draw(gen: torch.Generator, shape, dist: str, d: int) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) / math.sqrt(d)
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) / math.sqrt(d)
    if dist == "unit":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    raise ValueError(dist)


def make_inputs(w: Workload, B: int | None = None, H: int | None = None, T: int | None = None,
                seed: int | None = None):
    """Q, K [B,H,T,d] and V [B,H,T,dv] on the CPU in the workload's input type.
    B, H, T and seed may be overridden to draw a smaller case of the same recipe."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    q = _draw(gen, (B, H, T, w.d), w.qk_dist, w.d)
    k = _draw(gen, (B, H, T, w.d), w.qk_dist, w.d)
    v = _draw(gen, (B, H, T, w.dv), w.v_dist, w.d)
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def decode_tokens(w: DecodeWorkload = DECODE, n: int | None = None, count: int | None = None,
                  seed: int | None = None, device: str | torch.device = "cpu"):
    """Yields the decode stream token by token: for t = 0, 1, ... (prefill
    tokens first, then step tokens) the fp32 tensors q_t, k_t [n, d] and
    v_t [n, dv], drawn in that order from one generator.  ``device`` chooses
    where the generator runs (a CUDA generator gives a different stream with
    the same distribution; the parity tests use the CPU stream)."""
    n = w.n if n is None else n
    count = (w.prefill + w.steps) if count is None else count
    dist = "uniform" if w.normalized else "normal"
    gen = torch.Generator(device=device).manual_seed(w.seed if seed is None else seed)
    for _ in range(count):
        if device == "cpu":
            q = _draw(gen, (n, w.d), dist, w.d)
            k = _draw(gen, (n, w.d), dist, w.d)
            v = _draw(gen, (n, w.dv), "normal", w.d)
        else:
            q = _draw_on(gen, (n, w.d), dist, w.d, device)
            k = _draw_on(gen, (n, w.d), dist, w.d, device)
            v = _draw_on(gen, (n, w.dv), "normal", w.d, device)
        yield q, k, v


def _draw_on(gen, shape, dist, d, device):
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32, device=device) / math.sqrt(d)
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device) / math.sqrt(d)


def make_inputs_on(w: Workload, device, seed: int | None = None):
    """Same recipe as make_inputs, drawn by a generator on ``device`` (for
    timing runs whose inputs are too large to draw on the host quickly)."""
    gen = torch.Generator(device=device).manual_seed(w.seed if seed is None else seed)
    shp = (w.B, w.H, w.T)

    def draw(dim, dist):
        if dist == "uniform":
            x = torch.rand((*shp, dim), generator=gen, dtype=torch.float32, device=device) / math.sqrt(w.d)
        elif dist == "unit":
            x = torch.randn((*shp, dim), generator=gen, dtype=torch.float32, device=device)
        else:
            x = torch.randn((*shp, dim), generator=gen, dtype=torch.float32, device=device) / math.sqrt(w.d)
        return x.to(w.torch_dtype)

    q = draw(w.d, w.qk_dist)
    k = draw(w.d, w.qk_dist)
    v = draw(w.dv, w.v_dist)
    return q, k, v


def state_floats(d: int, dv: int) -> int:
    """Length of one head's decode-state record S|C|G|m|h in fp32 elements."""
    return d * d + 2 * d * dv + 2 * d
