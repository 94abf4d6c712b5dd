"""Row sharding across ranks.

Every row of the residual-add + RMSNorm forward depends only on itself (its
sum of squares covers its own hidden elements), so a batch splits across
GPUs by contiguous row blocks with no exchange at all: each rank runs the
op on its block, and the concatenation of the ranks' outputs is bit for bit
the single-GPU result.  This module only computes the split.
"""
from __future__ import annotations


def row_range(n_rows: int, rank: int, world: int) -> tuple[int, int]:
    """[lo, hi) rows of `rank` among `world` ranks: contiguous blocks, the
    first n_rows % world ranks taking one row more."""
    if world < 1 or not 0 <= rank < world or n_rows < 0:
        raise ValueError(f"bad split: n_rows={n_rows} rank={rank} world={world}")
    base, extra = divmod(n_rows, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def shard_rows(t, rank: int, world: int):
    """The rows of tensor `t` ([n_rows, ...]) that `rank` owns (a view)."""
    lo, hi = row_range(int(t.shape[0]), rank, world)
    return t[lo:hi]
