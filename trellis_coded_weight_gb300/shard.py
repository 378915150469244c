"""Row sharding of a packed trellis matrix across ranks (host logic only).

A stored row holds whole T-position blocks, so any split of the stored rows
keeps every block on one rank.  For an axis-1 layer (stored [out, in]) a row
shard computes a slice of the outputs, gathered along the output axis; for an
axis-0 layer (stored W^T [in, out]) a row shard holds a slice of the inputs
and produces a partial [M, out] sum, reduced across ranks.
"""
from __future__ import annotations


def row_range(rows: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, end) of stored rows owned by `rank`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_codes(codes, scales, rank: int, world: int):
    """This rank's rows of a packed matrix (codes [rows, words], scales [rows])."""
    s, e = row_range(codes.shape[0], rank, world)
    return codes[s:e], scales[s:e], (s, e)
