"""Multi-GPU decomposition of the projection: shard the batch, no collective.

Tokens of different batch elements never interact (the projection is
per-token, and rotary positions restart at every batch element), and the
fused weight is replicated, so N ranks each project a contiguous slice of the
batch and keep their outputs local. The only cross-rank step is host-side
bookkeeping: agreeing on the slowest rank's time.
"""
from __future__ import annotations

from typing import Tuple


def batch_shard(n_batch: int, rank: int, world: int) -> Tuple[int, int]:
    """[start, stop) of the batch elements rank `rank` of `world` projects.

    Contiguous, sizes differ by at most one, every element owned exactly once.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of {world}")
    base, extra = divmod(n_batch, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_view(x, batch_axis: int, rank: int, world: int):
    """A view (no copy) of x restricted to this rank's batch slice."""
    s, e = batch_shard(x.shape[batch_axis], rank, world)
    return x.narrow(batch_axis, s, e - s)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` across the default process group (the step time a
    multi-rank run reports); returns `value` when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
