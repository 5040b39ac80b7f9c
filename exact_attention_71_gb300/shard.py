"""Host-side sharding of attention work across ranks (one GPU per rank).

The work units of the forward pass, (batch, head, query tile), are
independent, so ranks take disjoint contiguous slices of the batch and never
exchange data on the path (weak scaling: per-rank work stays fixed as ranks
are added).
"""
from __future__ import annotations


def batch_shard(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the batch indices owned by `rank` (contiguous, sizes
    differing by at most one, every index owned exactly once)."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)
