"""Pins of the expert-cache oracle (oracle/cache.py): the pages' worked slot
split, byte-budget invariants, and hand-worked LRU sequences."""
import pytest

from oracle import cache as OC

MIB = 1 << 20


def test_plan_reproduces_the_pages_laguna_split():
    """FreeToken issue #194, Controlled A/B: the byte budget of 480 unified
    18 MiB slots holds 988 Q4_K (5.0625 MiB) + 202 BF16 (18 MiB) exact slots
    for 39 Q4_K and 8 BF16 layers at top-10."""
    budget = 480 * 18 * MIB
    q4k, bf16 = 3538944 + 1769472, 12582912 + 6291456      # per-expert bytes (Reproduction geometry)
    assert q4k == int(5.0625 * MIB) and bf16 == 18 * MIB
    assert OC.plan_slots(budget, [q4k, bf16], [39 * 10, 8 * 10]) == [988, 202]


def test_plan_invariants():
    for budget, b, w in [(10 ** 9, [3 * MIB, 7 * MIB, 11 * MIB], [30, 5, 1]), (7 * MIB - 1, [7 * MIB], [1]),
                         (123456789, [1000, 999], [1, 1000])]:
        n = OC.plan_slots(budget, b, w)
        used = sum(ni * bi for ni, bi in zip(n, b))
        assert used <= budget and budget - used < min(b)
    assert OC.plan_slots(100 * MIB, [7 * MIB], [3]) == [14]
    assert OC.plan_slots(7 * MIB - 1, [7 * MIB], [1]) == [0]


def test_lru_hand_worked_sequence():
    c = OC.SlotLRU(2)
    assert c.acquire(0, [5], 16) == ([0], [(0, 5)])           # never-used slots, lowest index first
    assert c.acquire(0, [7], 16) == ([1], [(1, 7)])
    assert c.acquire(0, [5], 16) == ([0], [])                 # hit: 5 becomes the most recent
    assert c.acquire(0, [9], 16) == ([1], [(1, 9)])           # evicts 7 (least recent)
    assert c.acquire(0, [7], 16) == ([0], [(0, 7)])           # evicts 5 (9 is more recent)
    assert c.acquire(1, [9, 9], 16) == ([1, 1], [(1, 9)])     # (layer 1, 9) is another key; a duplicate shares it
    assert c.acquire(0, [7, 20, -1], 16) == ([0, -1, -1], [])  # ids outside [0, E) get no slot
    assert (c.hits, c.misses) == (2, 5)


def test_lru_request_hits_are_never_evicted_by_its_misses():
    c = OC.SlotLRU(3)
    c.acquire(0, [1, 2, 3], 8)                                # slots 0, 1, 2; 1 is least recent
    out, fills = c.acquire(0, [4, 1], 8)                      # 1 is a hit, so 4 takes 2's slot (least recent left)
    assert out == [1, 0] and fills == [(1, 4)]
    with pytest.raises(ValueError):
        c.acquire(0, [1, 2, 3, 4], 8)


def test_lru_after_invalidation_keeps_the_order():
    """Hand-worked: 3 slots; [5, 6] fills slots 0 and 1 (order 2, 0, 1);
    after invalidation expert 5 misses and takes slot 2, the least recent --
    not slot 0, where it was, nor a reset order's slot 0."""
    lru = OC.SlotLRU(3)
    s, f = lru.acquire(0, [5, 6], 8)
    assert s == [0, 1] and f == [(0, 5), (1, 6)]
    lru.invalidate()
    s, f = lru.acquire(0, [5], 8)
    assert s == [2] and f == [(2, 5)]
    s, f = lru.acquire(0, [6, 5], 8)   # 5 hits; 6 misses and takes slot 0 (order was 0, 1, 2)
    assert s == [0, 2] and f == [(0, 6)]
    assert (lru.hits, lru.misses) == (1, 4)


def test_overlay_invalidates_exactly_the_overlapping_pools():
    a, b, c = OC.SlotLRU(2), OC.SlotLRU(2), OC.SlotLRU(2)
    arena = OC.Arena()
    arena.add_pool(a, [(0, 100), (100, 150)])
    arena.add_pool(b, [(150, 300)])
    arena.add_pool(c, [(300, 400)])
    for lru in (a, b, c):
        lru.acquire(0, [1], 4)
    assert arena.write_overlay(0, 150) == [0]      # ends where b starts: b keeps its tags
    assert arena.write_overlay(299, 300) == [1]    # one byte of b
    assert a.acquire(0, [1], 4)[1] == [(1, 1)]     # a forgot expert 1 (slot 1 was least recent)
    assert b.acquire(0, [1], 4)[1] == [(1, 1)]
    assert c.acquire(0, [1], 4)[1] == []           # c was never overlapped
