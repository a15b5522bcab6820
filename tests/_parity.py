"""Shared helpers for the GPU parity tests (tests only)."""
import os

import numpy as np
import torch

import oracle

# Tolerances, each max|o_gpu - o_ref| / max|o_ref| over the compared tensor:
TOL_TC_BF16 = 5e-3     # tensor-core paths with bf16 operands
TOL_NORMALIZED = 1e-4  # ratio-normalised variant
TOL_STEP_FP32 = 1e-5   # fp32 decode step
# The CUDA-core walks accumulate in fp32 from exact inputs; their error is
# fp32 rounding over the sequence (about 1e-6 here), held to this bound:
TOL_FP32_WALK = 1e-4

NTHREADS = max(1, min(16, os.cpu_count() or 1))


def relerr(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_forward(q, k, v, normalized=False):
    """Oracle outputs for CPU tensors [B,H,T,d] (any float dtype, upcast exactly)."""
    return oracle.serial(f64(q), f64(k), f64(v), normalized=normalized, nthreads=NTHREADS)


def forward_tolerance(dtype: torch.dtype, d: int, dv: int, normalized: bool) -> float:
    if normalized:
        return TOL_NORMALIZED
    return TOL_TC_BF16 if dtype == torch.bfloat16 else TOL_FP32_WALK
