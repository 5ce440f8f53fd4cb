"""Slot partition across GPUs: each rank owns one contiguous range of the
global slot space and holds the pool for it; requests are routed to the rank
that owns their slot.  Slots are independent, so no data moves between
ranks on the path (the only collective a caller may want is a gather of its
own outputs).  Host-side bookkeeping only, no arithmetic of the layer."""
from __future__ import annotations

import numpy as np


def slot_range(rank: int, world: int, n_slots: int) -> tuple[int, int]:
    """[lo, hi) of the global slots that `rank` owns (sizes differ by at most 1)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside [0, {world})")
    base, extra = divmod(n_slots, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def owner(slot: int, world: int, n_slots: int) -> int:
    """The rank that owns global slot `slot`."""
    if not 0 <= slot < n_slots:
        raise ValueError(f"slot {slot} outside [0, {n_slots})")
    base, extra = divmod(n_slots, world)
    cut = extra * (base + 1)
    return slot // (base + 1) if slot < cut else extra + (slot - cut) // base


def route(slot_ids, world: int, n_slots: int):
    """Split a batch of global slot ids by owner.  Returns, per rank, the
    positions of its entries in the batch and their slot ids local to that
    rank's pool (global id minus the range start)."""
    ids = np.asarray(slot_ids, dtype=np.int64)
    out = []
    for r in range(world):
        lo, hi = slot_range(r, world, n_slots)
        pos = np.nonzero((ids >= lo) & (ids < hi))[0]
        out.append((pos, (ids[pos] - lo).astype(np.int32)))
    return out
