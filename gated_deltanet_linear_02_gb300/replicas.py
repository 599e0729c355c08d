"""Timing across ranks when the mixer runs as independent replicas.

The mixer has no exchange step: sequences, layers and heads are independent
units, so N GPUs each run their own share of the work with no data-path
collective. The only cross-rank operations are timing plumbing: a barrier
around the timed region, and the maximum of the ranks' elapsed times. That
maximum is the job's time, because the job ends when the slowest rank ends.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def slowest_ms(local_ms: float, device=None) -> float:
    """The largest elapsed time over all ranks (local_ms when not distributed)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, job_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed, divided by the job's time."""
    if job_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return world * float(units_per_rank) / (job_ms / 1e3)
