"""Multi-GPU execution of the forward path: independent replicas.

Every (batch, head) of FAVOR+ attention is independent of every other, so N
GPUs run N independent problems (one process per GPU, each with its own
inputs) and nothing crosses between them on the data path.  The only
cross-rank step is the measurement: the job time is the slowest rank's time
and the job's work is the sum of every rank's work.
"""
from __future__ import annotations

__all__ = ["replica_seed", "job_aggregate"]


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s inputs: distinct per rank, reproducible."""
    return int(base_seed) + 1_000_003 * int(rank)


def job_aggregate(units: float, ms: float, group=None, device=None):
    """(total units over ranks, max ms over ranks); local values without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return float(units), float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(u.item()), float(t.item())
