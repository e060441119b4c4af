"""Oracle: the exact-geometry expert cache's host logic -- the split of a byte
budget into per-geometry slot pools and the LRU slot choice of each pool.

TEST INFRASTRUCTURE ONLY (see the package docstring).

FreeToken issue #194, "avoid max-stride padding for heterogeneous GGUF expert
banks", Proposed design: the byte-denominated bank arena is carved into
disjoint exact-width pools, one per geometry (tuple of row sizes), each with
its own tags and LRU state, decode views and LRU updates routed by layer.
Its Controlled A/B table gives the same byte budget as 480 unified 18 MiB
slots or as 988 Q4_K + 202 BF16 exact slots for Laguna-S (39 Q4_K layers of
5.0625 MiB experts, 8 BF16 layers of 18 MiB experts, top-10).

Readings (the pages print no rule):
  * plan: each geometry g gets slots in proportion to its routed expert
    selections per token, w_g = layers_g * top_k: n_g = floor(B * w_g /
    sum_h(w_h * bytes_h)); the bytes left over are then filled one slot at a
    time with the smallest expert size that still fits.  This reproduces the
    pages' 988 + 202.
  * LRU: a request (one layer's routed experts) first touches its hits, most
    recent last; each missing expert then takes the least recently used slot
    of the pool (never-used slots are the least recent, lowest index first)
    and becomes the most recent.  A request may not name more distinct
    experts than the pool has slots.  Keys are (layer, expert).

  * overlay: the full-layer prefill overlay is a byte range of the same
    arena as the pools (the pages: keep full-layer prefill on a shared
    overlay; invalidate the geometry pools before it is written).  Writing
    it invalidates every pool with a byte in that range -- each slot forgets
    its expert, the LRU order and the counters stay -- and no other pool.

Pins (tests/test_oracle_cache.py): the pages' 988 + 202 split; byte-budget
invariants; hand-worked LRU sequences, with and without invalidation; the
overlay's overlap rule on touching and overlapping ranges.
"""
from __future__ import annotations

from collections import OrderedDict


def plan_slots(budget_bytes: int, expert_bytes, selections) -> list[int]:
    """Slots per geometry for a byte budget (exact integer arithmetic)."""
    b = [int(v) for v in expert_bytes]
    w = [int(v) for v in selections]
    unit = sum(wi * bi for wi, bi in zip(w, b))
    n = [budget_bytes * wi // unit if unit > 0 else 0 for wi in w]
    left = budget_bytes - sum(ni * bi for ni, bi in zip(n, b))
    order = sorted(range(len(b)), key=lambda g: (b[g], g))
    while True:
        for g in order:
            if b[g] <= left:
                n[g] += 1
                left -= b[g]
                break
        else:
            return n


class SlotLRU:
    """One pool's slots and their LRU state."""

    def __init__(self, nslots: int):
        self.nslots = nslots
        self.order = OrderedDict((s, None) for s in range(nslots))   # least recent first
        self.key_of = [None] * nslots
        self.slot_of = {}
        self.hits = self.misses = 0

    def acquire(self, layer: int, ids, E: int):
        """Slots for one request's expert ids (-1 for ids outside [0, E));
        returns (slot per id, [(slot, expert) copied in, in order])."""
        keys = []
        for e in ids:
            k = (layer, int(e)) if 0 <= int(e) < E else None
            if k is not None and k not in keys:
                keys.append(k)
        if len(keys) > self.nslots:
            raise ValueError("more distinct experts than slots")
        for k in keys:
            if k in self.slot_of:
                self.order.move_to_end(self.slot_of[k])
                self.hits += 1
        fills = []
        for k in keys:
            if k in self.slot_of:
                continue
            s = next(iter(self.order))
            old = self.key_of[s]
            if old is not None:
                del self.slot_of[old]
            self.key_of[s] = k
            self.slot_of[k] = s
            self.order.move_to_end(s)
            self.misses += 1
            fills.append((s, k[1]))
        out = [self.slot_of[(layer, int(e))] if 0 <= int(e) < E else -1 for e in ids]
        return out, fills

    def invalidate(self):
        """Every slot forgets its expert; the LRU order and counters stay."""
        self.key_of = [None] * self.nslots
        self.slot_of = {}


class Arena:
    """Pools carved from one byte range, and the full-layer prefill overlay."""

    def __init__(self):
        self.pools = []   # (SlotLRU, [(lo, hi), ...]) in creation order

    def add_pool(self, lru: SlotLRU, ranges):
        self.pools.append((lru, [(int(a), int(b)) for a, b in ranges]))

    def write_overlay(self, lo: int, hi: int):
        """Invalidate the pools with a byte in [lo, hi), before the overlay
        is written; returns their indices in creation order."""
        hit = []
        for i, (lru, ranges) in enumerate(self.pools):
            if any(a < hi and lo < b for a, b in ranges):
                lru.invalidate()
                hit.append(i)
        return hit
