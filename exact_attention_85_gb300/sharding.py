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


def varlen_shard(cu_seqlens, world: int, rank: int):
    """Packed batch (device-independent prefix sums `cu_seqlens` of B
    sequences): the contiguous range of sequences owned by `rank`, chosen so
    that the ranks' attention work is balanced (proportional to n^2 per
    sequence, with or without the causal mask), and how to address it.

    Returns (seq_lo, seq_hi, row_lo, row_hi, local_cu): the rank owns
    sequences seq_lo .. seq_hi - 1, i.e. packed rows row_lo .. row_hi - 1, and
    `local_cu` are their prefix sums relative to row_lo (pass the slices
    [row_lo:row_hi] of the packed tensors and local_cu to the varlen entry
    points).  Sequences are never split, so no exchange is needed."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world size / rank")
    cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    lengths = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    work = [n * n for n in lengths]
    total = sum(work)
    # boundary r: first sequence whose cumulative work reaches r / world of the total
    bounds = [0]
    acc = 0
    i = 0
    for r in range(1, world):
        target = total * r / world
        while i < len(work) and acc + work[i] / 2 < target:
            acc += work[i]
            i += 1
        bounds.append(max(i, bounds[-1]))
    bounds.append(len(lengths))
    lo, hi = bounds[rank], bounds[rank + 1]
    row_lo, row_hi = cu[lo], cu[hi]
    local_cu = [c - row_lo for c in cu[lo:hi + 1]]
    return lo, hi, row_lo, row_hi, local_cu
