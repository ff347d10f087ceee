"""Host-side logic for running the SCAPE step on several GPUs.

Sharded split ("SCAPE" Sec. II-A: the distributed optimizer partitions the
parameters and optimizer states evenly over the workers; "Sintesi Tecnica:
SCAPE" Sec. 2: each worker computes the mask only for its own partition): rank
r of G owns the contiguous block of optimizer shards ``rank_shards(W, G, r)``
of one problem.  It holds a range handle (``Scape(..., shard_range=...)``, the
C ABI's ``scape_create_range``) over their parameter slice, with w, m and the
W residual rows of that slice only, and steps the slices of all W workers'
gradients there.  A shard's mask, packed values, synchronised buffer and
update depend only on its own slices, so with W workers simulated on every
GPU each rank draws its own gradient slices and the data path needs no
collective: the G ranks together step one problem of P parameters, each
holding about P/G of it.

The exchange a real data-parallel deployment needs, where each rank holds
only its own workers' full gradients, is in ``exchange.py``.
"""
from __future__ import annotations


def rank_shards(n_shards: int, world: int, rank: int) -> range:
    """Contiguous block of shards owned by `rank` (sizes differ by at most 1)."""
    if not (0 <= rank < world) or n_shards < 0:
        raise ValueError("bad rank/world/n_shards")
    return range(n_shards * rank // world, n_shards * (rank + 1) // world)


def shard_slice(P_global: int, W: int, shards: range) -> tuple:
    """Parameter range [lo, hi) of a block of shards of the even W-way split."""
    return shards.start * P_global // W, shards.stop * P_global // W


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


def sum_over_ranks(value: float, device=None) -> float:
    """Sum of `value` over all ranks of the default process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def weak_scaling_value(units_per_rank: int, world: int, t_max_s: float) -> float:
    """Whole-job throughput when every rank processes the same amount."""
    return units_per_rank * world / t_max_s


def strong_scaling_value(units_total: int, t_max_s: float) -> float:
    """Whole-job throughput of one problem split over the ranks: all the
    units, over the slowest rank's time."""
    return units_total / t_max_s


def gather_slices(local, lo: int, total: int):
    """Every rank contributes the slice [lo, lo + len(local)) of a vector of
    `total` elements (disjoint slices covering it); returns the whole vector
    on every rank.  CPU tensors (gloo) or device tensors (nccl)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local.clone()
    world = dist.get_world_size()
    meta = torch.tensor([lo, local.numel()], dtype=torch.int64, device=local.device)
    metas = [torch.empty_like(meta) for _ in range(world)]
    dist.all_gather(metas, meta)
    n_max = max(int(m[1]) for m in metas)
    pad = torch.zeros(n_max, dtype=local.dtype, device=local.device)
    pad[:local.numel()] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    out = torch.empty(total, dtype=local.dtype, device=local.device)
    for m, part in zip(metas, parts):
        a, n = int(m[0]), int(m[1])
        out[a:a + n] = part[:n]
    return out
