"""The expert cache on the GPU: three layers of one geometry share a pool of
12 slots; a sequence of requests (two or three tokens, top-4 of 32 experts)
misses, hits and evicts.  Each request decodes through the pool bank with
the slot ids moe_cache_acquire returns; its bf16 output must equal, bit for
bit, the same request decoded on the layer's fully resident bank (same
kernels on the same rows), the misses must follow the LRU oracle, and one
request is also checked against the layer oracle within the derived bounds."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import cache as OC  # noqa: E402
from oracle import formats as F  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from tests import cases  # noqa: E402
from tests import tolerance as tol  # noqa: E402

DEV = "cuda"


@pytest.mark.parametrize("pinned", [True, False])
def test_cache_decode_equals_resident_decode_and_follows_the_lru(pinned):
    """pinned: the layers' rows in pinned host memory (copied by the fill
    kernel over the host link) or in pageable memory (the copy engine)."""
    H, I, E, K, NSLOTS = 512, 256, 32, 4, 12
    wt = F.TYPE_Q4_K
    stream = torch.cuda.current_stream().cuda_stream
    # three layers, each with a request per token count; host copies of the
    # compact banks in pinned memory are the cache's source
    layers = []
    for l in range(3):
        reqs = [cases.make_case(H, I, E, K, wt, wt, T, seed=500 + 10 * l + T) for T in (2, 3)]
        src = reqs[0]
        pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
        host = dict(gu=pin(src.gu_dev.cpu()), dn=pin(src.dn_dev.cpu()), sb=pin(torch.from_numpy(src.sb.copy())))
        for rq in reqs[1:]:   # every request of a layer uses the first case's banks and scales
            rq.gu_dev, rq.dn_dev, rq.sb = src.gu_dev, src.dn_dev, src.sb
            rq.gu_rows, rq.dn_rows = src.gu_rows, src.dn_rows
        layers.append((reqs, host))
    geom = capi.moe_layer_geom(H, I, NSLOTS, K, wt, wt)
    cache = capi.moe_cache_create(geom, NSLOTS, stream)
    pool = capi.moe_cache_bank(cache)
    wsb = capi.moe_workspace_bytes(pool, 3)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    capi.moe_workspace_init(ws.data_ptr(), wsb, stream)
    lru = OC.SlotLRU(NSLOTS)
    order = [(0, 0), (1, 0), (0, 1), (2, 0), (1, 1), (2, 1), (0, 0), (1, 0)]
    checked_oracle = False
    for l, r in order:
        reqs, host = layers[l]
        case = reqs[r]
        T = case.x.shape[0]
        ids = [int(v) for v in case.ids.reshape(-1)]
        slots, nfill = capi.moe_cache_acquire(cache, l, host["gu"].data_ptr(), host["dn"].data_ptr(),
                                              host["sb"].data_ptr(), E, ids, stream)
        want_slots, fills = lru.acquire(l, ids, E)
        assert slots == want_slots and nfill == len(fills)
        x = torch.from_numpy(case.x.view(np.int16)).to(DEV)
        sid = torch.tensor(slots, dtype=torch.int32, device=DEV).reshape(T, K)
        w = torch.from_numpy(case.w).to(DEV)
        out = torch.empty((T, H), dtype=torch.int16, device=DEV)
        capi.moe_decode(pool, x.data_ptr(), T, sid.data_ptr(), w.data_ptr(), out.data_ptr(), ws.data_ptr(), wsb,
                        stream)
        torch.cuda.synchronize()
        got = out.cpu().numpy().view(np.uint16)
        assert capi.moe_get_error(ws.data_ptr(), wsb, stream) == 0
        direct = cases.run_gpu(case, stages=False)
        assert np.array_equal(got, direct["out"]), (l, r)
        if not checked_oracle and r == 0 and nfill > 0:   # the first case of a layer holds all its routed rows
            ref, _, st = cases.oracle(case)
            beta, _, _ = tol.output_bounds(case.geom, st)
            tol.check_output(got, ref, beta)
            checked_oracle = True
    hits, misses, copied = capi.moe_cache_stats(cache)
    assert (hits, misses) == (lru.hits, lru.misses) and misses > NSLOTS   # slots were reused
    rb_gu, rb_dn = F.row_bytes(wt, H), F.row_bytes(wt, I)
    assert copied == misses * (2 * I * rb_gu + H * rb_dn + 16)
    capi.moe_cache_destroy(cache)
