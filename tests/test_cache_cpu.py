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
