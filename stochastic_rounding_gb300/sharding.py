"""Host-side planning of a sharded optimizer step.

Because every element's random bits depend only on (seed, step, global
parameter position), the flattened parameter vector can be split into
contiguous ranges, one per rank, and each rank updates its range with no
communication inside the step ("adamw-sr", Method: identical whether a
parameter is updated whole or split across shards and ranks).  These helpers
compute the ranges and, for one rank, the per-tensor pieces it owns with the
base_index each piece must carry.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def shard_bounds(total: int, world: int, rank: int, align: int = 4) -> Tuple[int, int]:
    """[start, end) of rank's contiguous share of ``total`` elements.  Cut
    points are multiples of ``align`` (so shards keep the vectorised path)
    except for the final end; shares differ by at most ``align`` elements."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if align < 1:
        raise ValueError("align must be >= 1")
    units = -(-total // align)
    lo = units * rank // world
    hi = units * (rank + 1) // world
    return min(total, lo * align), min(total, hi * align)


def shard_pieces(sizes: Sequence[int], start: int, end: int) -> List[Tuple[int, int, int, int]]:
    """The parts of tensors (laid out back to back in ``sizes`` order) that
    fall in the global range [start, end): (tensor, local offset, length,
    base_index) with base_index = global position of the piece's element 0."""
    out = []
    pos = 0
    for t, n in enumerate(sizes):
        a, b = max(start, pos), min(end, pos + n)
        if a < b:
            out.append((t, a - pos, b - a, a))
        pos += n
    return out
