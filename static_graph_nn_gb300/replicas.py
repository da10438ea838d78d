"""Replica bookkeeping for the benchmark under torchrun: the training step has
no exchange between GPUs (replicas only), so each rank runs its own copy and
the job's time is the slowest rank's; the job's throughput is the steps of all
ranks over that time."""
from __future__ import annotations


def max_over_ranks(values: list[float], device=None) -> list[float]:
    """Elementwise maximum of `values` across all ranks (identity without a
    process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, steps_per_rank: int, seconds: float) -> float:
    """Steps per second of the whole job: every rank ran steps_per_rank steps."""
    return world * steps_per_rank / seconds
