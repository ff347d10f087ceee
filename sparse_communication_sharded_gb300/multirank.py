"""Host-side logic for running the SCAPE step on several GPUs.

Optimizer shards are independent: a shard's mask, packed buffers, reduce and
update depend only on that shard's slices of the W workers' gradients (plus the
global step count).  So ranks split work by whole shards and exchange nothing
on the data path; the only collectives are the measurement's barrier and the
max over ranks of the step time.
"""
from __future__ import annotations


def rank_shards(n_shards: int, world: int, rank: int) -> range:
    """Contiguous block of shards owned by `rank` (sizes differ by at most 1)."""
    if not (0 <= rank < world) or n_shards < 0:
        raise ValueError("bad rank/world/n_shards")
    return range(n_shards * rank // world, n_shards * (rank + 1) // world)


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks of the default process group (the value
    itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank: int, world: int, t_max_s: float) -> float:
    """Whole-job throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / t_max_s
