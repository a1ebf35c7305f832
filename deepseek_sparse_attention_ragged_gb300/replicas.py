"""Replica aggregation for running the decode on N GPUs of one node.

Rows are independent and every GPU holds whole rows, so N GPUs run N
replicas of the step with no data-path collective. The only cross-rank
operations are the timing barrier and the maximum of the ranks' times, which
decide the job's rate: the slowest replica bounds the whole job.
"""

from __future__ import annotations

import torch


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of `x` over the ranks of the default process group (x when
    there is no group). The tensor lives on `device` for NCCL, on the host for
    gloo."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    on_host = dist.get_backend() == "gloo"
    t = torch.tensor([float(x)], dtype=torch.float64, device="cpu" if on_host else device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, rows_per_replica: int, steps: int, total_ms: float) -> float:
    """Rows per second of the whole job: every replica advances its rows by
    `steps` steps, and the job takes the slowest replica's `total_ms`."""
    if total_ms <= 0:
        raise ValueError("total_ms must be positive")
    return world * rows_per_replica * steps / (total_ms / 1e3)
