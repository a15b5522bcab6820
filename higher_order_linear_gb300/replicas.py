"""Host-side helpers for running the forward as independent replicas, one
per GPU (heads are independent; the path needs no data exchange).

Only timing crosses ranks: every rank times its own replica, the slowest rank
sets the job time, and the job throughput is all ranks' units over that time.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def head_range(BH: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced split of BH heads over `world` ranks: rank r owns
    heads [begin, end).  Used when one batch is spread over ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    return BH * rank // world, BH * (rank + 1) // world


def max_over_ranks(x: float, device: torch.device | str = "cpu") -> float:
    """Maximum of a per-rank float over the default process group (identity
    when torch.distributed is not initialised)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank processed units_per_rank
    in at most ms_max milliseconds."""
    if ms_max <= 0:
        raise ValueError("time must be positive")
    return world * units_per_rank / (ms_max / 1e3)
