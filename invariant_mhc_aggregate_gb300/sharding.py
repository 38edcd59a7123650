"""Token sharding for data-parallel use on several GPUs.

The operation is independent per token: the forward, grad_residual and the
ORDER-256 grad_pre of a token depend on that token's bytes and on H only.  A
batch therefore splits into contiguous token ranges, one per GPU, with no
exchange between them, and the concatenated results are byte-identical to a
single call over the whole batch.
"""

from __future__ import annotations


def token_range(T: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the tokens rank `rank` of `world` owns: contiguous ranges,
    the first T % world ranks one token longer."""
    if world <= 0 or not 0 <= rank < world or T < 0:
        raise ValueError(f"bad shard request T={T} rank={rank} world={world}")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)
