"""Host-side logic of multi-process runs (one process per GPU).

The indexer path shards by rows: every rank scores and selects its own batch
with no data-path exchange (weak scaling).  Only the timing is combined: the
job's step time is the slowest rank's.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own synthetic batch (distinct per rank, rank 0 keeps the base seed)."""
    return seed + 1000 * rank


def job_step_ms(local_ms: float, device=None) -> float:
    """Max over ranks of the per-step time (the job is as fast as its slowest rank)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, step_ms: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed per second."""
    return units_per_rank * world / (step_ms * 1e-3)
