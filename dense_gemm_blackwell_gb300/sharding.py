"""Partition one product over ranks with no collective on the data path.

D = A * B^T splits into independent output blocks: the rank that owns rows
[m0, m1) of A computes rows [m0, m1) of D from the whole of B, and a batched
problem splits along its batch.  No rank reads another rank's result, so the
only cross-rank operations a job needs are for measurement (a barrier and the
maximum of the ranks' times).  Shards are contiguous and aligned to the MMA
tile height so that each rank's tiles are full tiles except at the end of M.
"""
from __future__ import annotations


def row_shard(M: int, world: int, rank: int, align: int = 256) -> tuple[int, int]:
    """Rows [m0, m1) of D owned by `rank`: contiguous, aligned to `align`, balanced."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    blocks = (M + align - 1) // align
    b0 = blocks * rank // world
    b1 = blocks * (rank + 1) // world
    return min(M, b0 * align), min(M, b1 * align)


def batch_shard(batch: int, world: int, rank: int) -> tuple[int, int]:
    """Batch entries [b0, b1) owned by `rank`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    return batch * rank // world, batch * (rank + 1) // world
