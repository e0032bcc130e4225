"""Data-parallel sharding of a decode batch across ranks.

Tokens are independent: every output row depends only on its own token's routes, residual row and
the shared gamma (RMSNorm is row-local), so a batch splits across GPUs by token with no collective.
Each rank runs the fused finalize on its contiguous token range.
"""
from __future__ import annotations


def token_range(T: int, rank: int, world: int) -> tuple[int, int]:
    """[t0, t1) of rank `rank` out of `world`: contiguous, sizes differing by at most one, in rank order."""
    if world < 1 or not (0 <= rank < world) or T < 0:
        raise ValueError(f"bad shard request T={T} rank={rank} world={world}")
    base, extra = divmod(T, world)
    t0 = rank * base + min(rank, extra)
    return t0, t0 + base + (1 if rank < extra else 0)
