"""The expert cache's host logic in the library against the oracle
(oracle/cache.py), without a GPU: the byte-budget split into exact-geometry
pools and the LRU slot choice of a pool, request by request."""
import os

import numpy as np
import pytest

from oracle import cache as OC

MIB = 1 << 20


@pytest.fixture(scope="module")
def capi():
    from quantized_routed_expert_route_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    from quantized_routed_expert_route_gb300 import capi as c
    return c


def test_plan_matches_the_oracle_and_the_pages(capi):
    q4k, bf16 = 3538944 + 1769472, 12582912 + 6291456
    assert capi.moe_cache_plan(480 * 18 * MIB, [q4k, bf16], [390, 80]) == [988, 202]
    r = np.random.default_rng(0)
    for _ in range(200):
        g = int(r.integers(1, 5))
        b = [int(v) for v in r.integers(1000, 50 * MIB, size=g)]
        w = [int(v) for v in r.integers(0, 500, size=g)]
        budget = int(r.integers(0, 1 << 36))
        assert capi.moe_cache_plan(budget, b, w) == OC.plan_slots(budget, b, w), (budget, b, w)


def test_slot_table_matches_the_oracle_lru(capi):
    r = np.random.default_rng(1)
    for nslots, E in [(6, 16), (1, 4), (12, 40)]:
        t = capi.SlotTable(nslots)
        o = OC.SlotLRU(nslots)
        for _ in range(400):
            layer = int(r.integers(0, 3))
            n = int(r.integers(0, nslots + 3))
            ids = [int(v) for v in r.integers(-2, E + 2, size=n)]
            try:
                want = o.acquire(layer, ids, E)
            except ValueError:
                with pytest.raises(capi.MoeError) as ei:
                    t.acquire(layer, ids, E)
                assert ei.value.status == capi.MOE_EUNSUPPORTED
                continue
            assert t.acquire(layer, ids, E) == want, (layer, ids)
        assert t.stats() == (o.hits, o.misses)
        t.close()


def test_slot_table_invalidation_matches_the_oracle(capi):
    """Requests interleaved with invalidations (the full-layer prefill
    overlay's first step): the library's slot choices, copies and counters
    follow the oracle's, which keeps the LRU order across an invalidation."""
    r = np.random.default_rng(2)
    for nslots, E in [(5, 12), (2, 3), (16, 64)]:
        t = capi.SlotTable(nslots)
        o = OC.SlotLRU(nslots)
        for _ in range(300):
            if r.random() < 0.1:
                t.invalidate()
                o.invalidate()
                continue
            layer = int(r.integers(0, 2))
            n = int(r.integers(0, nslots + 1))
            ids = [int(v) for v in r.integers(-1, E + 1, size=n)]
            try:
                want = o.acquire(layer, ids, E)
            except ValueError:
                continue
            assert t.acquire(layer, ids, E) == want, (layer, ids)
        assert t.stats() == (o.hits, o.misses)
        t.close()


def test_carved_pool_and_overlay_sizes(capi):
    """Host-side sizing and argument checks of carved pools and the overlay
    (no device memory is touched)."""
    import ctypes
    q4k = capi.moe_layer_geom(512, 256, 32, 4, capi.MOE_Q4_K, capi.MOE_Q4_K)
    rb = capi.moe_row_bytes(capi.MOE_Q4_K, 512), capi.moe_row_bytes(capi.MOE_Q4_K, 256)
    gu, dn = 2 * 256 * rb[0], 512 * rb[1]

    def a256(v):
        return (v + 255) // 256 * 256
    assert capi.moe_cache_bytes(q4k, 12) == a256(12 * gu + 256) + a256(12 * dn + 256)
    assert capi.moe_overlay_bytes(q4k) == a256(32 * gu + 256) + a256(32 * dn + 256)
    assert capi.moe_cache_bytes(q4k, 0) == 0
    lib = capi.library()
    out = ctypes.c_void_p()
    assert lib.moe_cache_create_at(ctypes.byref(q4k), 12, None, 1 << 30, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_cache_create_at(ctypes.byref(q4k), 12, 256 + 16, 1 << 30, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_cache_create_at(ctypes.byref(q4k), 12, 4096, 100, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_overlay_create(ctypes.byref(q4k), 4096, 100, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_overlay_load(None, None, 0, None, None, None, None) == capi.MOE_EINVAL
    assert lib.moe_cache_invalidate(None) == capi.MOE_EINVAL
    assert lib.moe_overlay_destroy(None) == capi.MOE_OK
