"""Batch sharding across ranks (one process per GPU).

Each sequence carries its own fast-weight state that starts from W_down0
(reset at document boundaries, "[논문리뷰] In-Place Test-Time Training",
Method §3), so sequences are independent units: a rank runs the layer on its
contiguous share of the batch and no tensor crosses ranks.  The only
cross-rank traffic is host-side bookkeeping: barriers and the max of the
ranks' timings.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_range(total: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of `rank`'s contiguous share of `total` units; shares
    differ by at most one unit and cover every unit exactly once."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device: torch.device | None = None) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank's);
    the value itself when no process group is running."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device: torch.device | None = None) -> None:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()
