"""Host-side plan for running the layer on several GPUs, one process per GPU.

The sparse linear layer splits with no exchange along N (output channels):
each rank owns a contiguous block of weight rows, compresses only those rows
and multiplies them with the full activation, producing a disjoint block of
Y's columns.  Splitting M (tokens) replicates the weight instead.  Neither
needs a collective on the data path; gathering Y on one rank is the caller's
choice, not part of the layer.

Blocks are whole 128-row tiles so every shard is a valid GEMM operand and the
per-channel / 128x128 weight scales of a shard are exactly the unsharded
scales restricted to its rows.
"""
from typing import List, Tuple

TILE_ROWS = 128


def shard_rows(N: int, world: int, rank: int) -> Tuple[int, int]:
    """[begin, end) weight rows owned by `rank`: whole 128-row tiles, spread
    as evenly as possible (the first N/128 % world ranks get one more)."""
    if N % TILE_ROWS != 0:
        raise ValueError("N must be a multiple of %d" % TILE_ROWS)
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    tiles = N // TILE_ROWS
    base, extra = divmod(tiles, world)
    begin = rank * base + min(rank, extra)
    count = base + (1 if rank < extra else 0)
    return begin * TILE_ROWS, (begin + count) * TILE_ROWS


def shard_plan(N: int, world: int) -> List[Tuple[int, int]]:
    return [shard_rows(N, world, r) for r in range(world)]


def aggregate_throughput(units_per_rank: float, seconds_per_rank: List[float]) -> float:
    """Whole-job throughput: all units processed by all ranks over the slowest
    rank's time (every rank runs the same work; the job ends with the last)."""
    return units_per_rank * len(seconds_per_rank) / max(seconds_per_rank)
