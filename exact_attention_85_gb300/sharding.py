"""Data-parallel sharding of the attention path across ranks (one GPU each).

The unit of work is a (batch, key/value-head group) pair: one key/value head
together with the Hq / Hkv query heads that read it.  Forward and backward of
one unit touch no data of another unit (the grouped dK / dV sums stay inside
the unit), so ranks that own disjoint units need no exchange step at all: no
collective appears on the data path.  Only timing (a barrier and the maximum
of the step times) is combined across ranks.

`unit_range` splits the B * Hkv units of a global problem into contiguous,
nearly equal blocks, one per rank (strong scaling).  The benchmark runs the
weak-scaling form: every rank owns a full per-GPU batch of its own.
"""
from __future__ import annotations


def unit_range(B: int, Hkv: int, world: int, rank: int) -> tuple[int, int]:
    """Half-open range [lo, hi) of flat unit indices u = b * Hkv + g owned by
    `rank`; the first (B * Hkv) % world ranks get one extra unit."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world size / rank")
    total = B * Hkv
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def units(B: int, Hkv: int, world: int, rank: int) -> list[tuple[int, int]]:
    """(batch, kv-head) pairs owned by `rank`."""
    lo, hi = unit_range(B, Hkv, world, rank)
    return [divmod(u, Hkv) for u in range(lo, hi)]


def query_heads(g: int, Hq: int, Hkv: int) -> range:
    """Query heads that read key/value head g (consecutive heads share one)."""
    G = Hq // Hkv
    return range(g * G, (g + 1) * G)
