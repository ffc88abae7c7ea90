"""Host-side sharding of independent work across ranks (one GPU per rank).

Diversity sequences are independent of one another, and so are BMU samples:
a batch splits across ranks with no exchange on the data path.  Each rank
runs its contiguous share through the library on its own GPU; the results
are gathered on the host afterwards (`gather_rows`), which is the only
collective and carries outputs, not operands.
"""
from __future__ import annotations


def shard_range(total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of `total` items for `rank` of `world`;
    the first `total % world` ranks take one extra item."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if total < 0:
        raise ValueError("total must be >= 0")
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_rows(local, group=None):
    """Concatenate every rank's rows (a numpy array or CPU tensor with the
    same trailing shape) in rank order, on every rank."""
    import numpy as np
    import torch
    import torch.distributed as dist

    arr = local.numpy() if isinstance(local, torch.Tensor) else np.asarray(local)
    world = dist.get_world_size(group)
    parts = [None] * world
    dist.all_gather_object(parts, arr, group=group)
    return np.concatenate(parts, axis=0)
