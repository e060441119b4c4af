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
from synth import banks as S  # noqa: E402
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


def test_prefill_overlay_invalidates_the_pools_it_overwrites():
    """One arena: an NVFP4 pool (4 slots) at its start, inside the region of
    the full-layer prefill overlay, and a Q8_0 pool (2 slots) after it.
    Decoding through the NVFP4 pool equals resident decoding; loading the
    layer into the overlay invalidates that pool (it overwrote its slots) but
    not the Q8_0 pool; prefill on the overlay bank equals prefill on the
    resident bank bit for bit (fixed-order W4A4); the same decode request
    through the NVFP4 pool then misses every expert again and still equals
    resident decoding, while the Q8_0 pool's request hits."""
    H, I, E, K, T = 256, 256, 8, 2, 2
    nv = capi.MOE_NVFP4
    stream = torch.cuda.current_stream().cuda_stream
    case = cases.make_prefill_case(H, I, E, K, 64, seed=910)
    gu_host = case.gu_dev.cpu().pin_memory()
    dn_host = case.dn_dev.cpu().pin_memory()
    sb_dev = torch.from_numpy(case.sb).to(DEV)
    sb_host = torch.from_numpy(case.sb.copy()).pin_memory()
    geom = capi.moe_layer_geom(H, I, E, K, nv, nv)
    resident = capi.moe_bank_create(geom, case.gu_dev.data_ptr(), case.gu_dev.numel(), case.dn_dev.data_ptr(),
                                    case.dn_dev.numel(), sb_dev.data_ptr(), capi.MOE_SRC_DEVICE_BORROW, stream)
    q8 = cases.make_case(H, I, E, K, F.TYPE_Q8_0, F.TYPE_Q8_0, T, seed=911)
    q8_gu, q8_dn = q8.gu_dev.cpu().pin_memory(), q8.dn_dev.cpu().pin_memory()
    # the arena: [overlay region, with the NVFP4 pool at its start][the Q8_0 pool]
    ov_bytes = capi.moe_overlay_bytes(geom)
    pa_bytes = capi.moe_cache_bytes(geom, 4)
    g8 = capi.moe_layer_geom(H, I, E, K, capi.MOE_Q8_0, capi.MOE_Q8_0)
    pb_bytes = capi.moe_cache_bytes(g8, 2)
    assert pa_bytes < ov_bytes
    arena = torch.empty(ov_bytes + pb_bytes, dtype=torch.uint8, device=DEV)
    base = arena.data_ptr()
    assert base % 256 == 0
    pool_a = capi.moe_cache_create_at(geom, 4, base, pa_bytes, stream)
    pool_b = capi.moe_cache_create_at(g8, 2, base + ov_bytes, pb_bytes, stream)
    overlay = capi.moe_overlay_create(geom, base, ov_bytes, stream)
    bank_a = capi.moe_cache_bank(pool_a)
    wsb = max(capi.moe_workspace_bytes(bank_a, T), capi.moe_workspace_bytes(resident, T))
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    capi.moe_workspace_init(ws.data_ptr(), wsb, stream)
    x = torch.from_numpy(S.hidden_bf16(912, T, H).view(np.int16)).to(DEV)
    ids_np = np.array([[1, 5], [5, 6]], dtype=np.int32)
    w = torch.tensor([[0.6, 0.4], [0.3, 0.7]], dtype=torch.float32, device=DEV)

    def decode(bank, ids):
        out = torch.empty((T, H), dtype=torch.int16, device=DEV)
        capi.moe_decode(bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), out.data_ptr(), ws.data_ptr(), wsb,
                        stream)
        torch.cuda.synchronize()
        assert capi.moe_get_error(ws.data_ptr(), wsb, stream) == 0
        return out.cpu().numpy().view(np.uint16)

    want = decode(resident, torch.from_numpy(ids_np).to(DEV))

    def through_pool():
        slots, nfill = capi.moe_cache_acquire(pool_a, 0, gu_host.data_ptr(), dn_host.data_ptr(), sb_host.data_ptr(),
                                              E, [int(v) for v in ids_np.reshape(-1)], stream)
        got = decode(bank_a, torch.tensor(slots, dtype=torch.int32, device=DEV).reshape(T, K))
        return got, nfill

    got, nfill = through_pool()
    assert nfill == 3 and np.array_equal(got, want)
    got, nfill = through_pool()
    assert nfill == 0 and np.array_equal(got, want)          # all hits
    _, nb = capi.moe_cache_acquire(pool_b, 0, q8_gu.data_ptr(), q8_dn.data_ptr(), None, E, [2, 3], stream)
    assert nb == 2
    # the overlay: invalidates pool_a (it lies inside), not pool_b, then copies the layer in
    capi.moe_overlay_load(overlay, [pool_a, pool_b], gu_host.data_ptr(), dn_host.data_ptr(), sb_host.data_ptr(),
                          stream)
    Tp = case.x.shape[0]
    xp = torch.from_numpy(case.x.view(np.int16)).to(DEV)
    idp, wp = torch.from_numpy(case.ids).to(DEV), torch.from_numpy(case.w).to(DEV)
    mode = capi.MOE_PREFILL_W4A4_FIXED

    def prefill(bank):
        pw = capi.moe_prefill_workspace_bytes(bank, Tp, mode)
        pws = torch.empty(pw, dtype=torch.uint8, device=DEV)
        out = torch.empty((Tp, H), dtype=torch.int16, device=DEV)
        capi.moe_prefill_grouped(bank, xp.data_ptr(), Tp, idp.data_ptr(), wp.data_ptr(), mode, out.data_ptr(),
                                 pws.data_ptr(), pw, stream)
        torch.cuda.synchronize()
        assert capi.moe_get_error(pws.data_ptr(), pw, stream) == 0
        return out.cpu().numpy().view(np.uint16)

    assert np.array_equal(prefill(capi.moe_overlay_bank(overlay)), prefill(resident))
    # pool_a's slots were overwritten and forgotten: every expert is copied again
    got, nfill = through_pool()
    assert nfill == 3 and np.array_equal(got, want)
    _, nb = capi.moe_cache_acquire(pool_b, 0, q8_gu.data_ptr(), q8_dn.data_ptr(), None, E, [2, 3], stream)
    assert nb == 0
    torch.cuda.synchronize()
    capi.moe_overlay_destroy(overlay)
    capi.moe_cache_destroy(pool_a)
    capi.moe_cache_destroy(pool_b)
    capi.moe_bank_destroy(resident)
