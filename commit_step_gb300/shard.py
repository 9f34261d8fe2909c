"""Batch-row sharding of the commit step across ranks.

Every statistic is per row and every commit rule is per batch row, so a
batch split by batch rows needs no exchange: rank r takes batch rows
[b0, b1) and computes them alone (weak scaling when each rank brings its own
batch).  No collective is involved in the data path.
"""
from __future__ import annotations


def shard_batch_rows(B: int, rank: int, world: int):
    """Contiguous, balanced [b0, b1) of batch rows for `rank` of `world`."""
    if world <= 0 or not (0 <= rank < world) or B < 0:
        raise ValueError("bad shard request")
    return (B * rank) // world, (B * (rank + 1)) // world
