"""Seeded decode cases shared by the GPU tests: banks on the device (counter
filler everywhere, converted rows for the routed experts), the same routed
rows on the host for the oracle, and the runner that exports the stages."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from oracle import formats as F
from oracle import layer as OL
from synth import banks as S
from synth import counter as C


@dataclass
class Case:
    geom: OL.Geometry
    x: np.ndarray          # uint16 [T, H]
    ids: np.ndarray        # int32 [T, K]
    w: np.ndarray          # fp32 [T, K]
    sb: np.ndarray         # fp32 [E, 4]
    gu_rows: dict          # expert -> uint8 [2I, rb]
    dn_rows: dict          # expert -> uint8 [H, rb]
    gu_dev: object = None  # torch uint8 CUDA tensors holding the whole banks
    dn_dev: object = None


def make_case(H, I, E, K, gu_t, dn_t, T, seed, routing="softmax", ids=None, device="cuda", glu=0) -> Case:
    import torch
    if ids is None:
        if routing == "zipf":
            ids, w = S.zipf_routing(seed + 2, T, E, K)
        else:
            ids, w = S.softmax_topk_routing(seed + 2, T, E, K)
    else:
        ids = np.asarray(ids, dtype=np.int32).reshape(T, K)
        w = S.rng(seed + 3).uniform(0.05, 1.0, size=(T, K)).astype(np.float32)
    x = S.hidden_bf16(seed + 1, T, H)
    sb = S.counter_scale_bank(seed + 4, E, gu_t, dn_t)
    routed = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < E})
    gu_rows, dn_rows = {}, {}
    for e in routed:
        gu_rows[e], dn_rows[e], sb[e] = S.converted_expert(seed, e, H, I, gu_t, dn_t)
    rb_gu, rb_dn = F.row_bytes(gu_t, H), F.row_bytes(dn_t, I)
    gu_dev = torch.empty(E * 2 * I * rb_gu + 16, dtype=torch.uint8, device=device)
    dn_dev = torch.empty(E * H * rb_dn + 16, dtype=torch.uint8, device=device)
    n_gu, n_dn = E * 2 * I * rb_gu, E * H * rb_dn
    if n_gu % 8 == 0 and n_dn % 8 == 0:
        C.fill_bank_torch(gu_dev[:n_gu], seed * 31 + 5, gu_t, H)
        C.fill_bank_torch(dn_dev[:n_dn], seed * 31 + 6, dn_t, I)
    else:
        gu_dev[:n_gu].copy_(torch.from_numpy(C.bank_bytes_np(seed * 31 + 5, gu_t, H, 0, E * 2 * I).reshape(-1)))
        dn_dev[:n_dn].copy_(torch.from_numpy(C.bank_bytes_np(seed * 31 + 6, dn_t, I, 0, E * H).reshape(-1)))
    for e in routed:
        gu_dev[e * 2 * I * rb_gu:(e + 1) * 2 * I * rb_gu].copy_(torch.from_numpy(gu_rows[e].reshape(-1)))
        dn_dev[e * H * rb_dn:(e + 1) * H * rb_dn].copy_(torch.from_numpy(dn_rows[e].reshape(-1)))
    return Case(OL.Geometry(H, I, E, K, gu_t, dn_t, glu), x, ids, w, sb, gu_rows, dn_rows,
                gu_dev[:n_gu], dn_dev[:n_dn])


def oracle(case: Case, tokens=None):
    """Oracle output (fp64 [T', H]) and stages for all tokens or a sample."""
    sel = np.arange(case.x.shape[0]) if tokens is None else np.asarray(tokens)
    return OL.moe_layer(case.geom, case.gu_rows, case.dn_rows, case.sb, case.x[sel], case.ids[sel],
                        case.w[sel], stages=True)


def run_gpu(case: Case, stages=True):
    """Decode on the GPU through the C ABI; returns numpy results."""
    import torch

    from quantized_routed_expert_route_gb300 import capi
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    T = case.x.shape[0]
    dev = "cuda"
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to(dev), borrow=True, max_tokens=max(T, 1), glu=g.glu)
    x = torch.from_numpy(case.x.view(np.int16)).to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    w = torch.from_numpy(case.w).to(dev)
    out = torch.empty((T, g.H), dtype=torch.int16, device=dev)
    res = {}
    stream = torch.cuda.current_stream().cuda_stream
    if stages and T <= capi.MOE_DECODE_T_CHUNK and T > 0:
        RT = T * g.top_k
        xb = torch.zeros((T, g.H // 32 * 36), dtype=torch.uint8, device=dev)
        inter = torch.zeros((RT, g.I), dtype=torch.float32, device=dev)
        ib = torch.zeros((RT, g.I // 32 * 36), dtype=torch.uint8, device=dev)
        capi.moe_debug_decode_stages(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), out.data_ptr(),
                                     layer.ws.data_ptr(), layer.ws_bytes, stream, xb.data_ptr(),
                                     inter.data_ptr(), ib.data_ptr())
        torch.cuda.synchronize()
        res["x_blocks"] = xb.cpu().numpy()
        res["inter"] = inter.cpu().numpy().reshape(T, g.top_k, g.I)
        res["inter_blocks"] = ib.cpu().numpy().reshape(T, g.top_k, g.I // 32, 36)
    else:
        capi.moe_decode(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), out.data_ptr(),
                        layer.ws.data_ptr(), layer.ws_bytes, stream)
        torch.cuda.synchronize()
    res["out"] = out.cpu().numpy().view(np.uint16)
    res["err"] = layer.error_bits()
    res["launches"] = capi.moe_decode_kernel_count(layer.bank, T)
    layer.close()
    return res


# ------------------------------------------------------------------ prompt path

@dataclass
class PrefillCase:
    geom: OL.Geometry
    x: np.ndarray          # uint16 [T, H]
    ids: np.ndarray        # int32 [T, K]
    w: np.ndarray          # fp32 [T, K]
    sb: np.ndarray         # fp32 [E, 4]
    seed: int
    gu_dev: object = None
    dn_dev: object = None


def make_prefill_case(H, I, E, K, T, seed, routing="softmax", ids=None, device="cuda", glu=0) -> PrefillCase:
    """NVFP4 banks filled on the device by the counter-based generator (every
    expert is routed to in a prompt chunk); the oracle regenerates the rows of
    the experts it checks on the host."""
    import torch
    if ids is None:
        if routing == "zipf":
            ids, w = S.zipf_routing(seed + 2, T, E, K)
        else:
            ids, w = S.softmax_topk_routing(seed + 2, T, E, K)
    else:
        ids = np.asarray(ids, dtype=np.int32).reshape(T, K)
        w = S.rng(seed + 3).uniform(0.05, 1.0, size=(T, K)).astype(np.float32)
    x = S.hidden_bf16(seed + 1, T, H)
    t = F.TYPE_NVFP4
    sb = S.counter_scale_bank(seed + 4, E, t, t)
    rb_gu, rb_dn = F.row_bytes(t, H), F.row_bytes(t, I)
    n_gu, n_dn = E * 2 * I * rb_gu, E * H * rb_dn
    gu_dev = torch.empty(n_gu + 16, dtype=torch.uint8, device=device)
    dn_dev = torch.empty(n_dn + 16, dtype=torch.uint8, device=device)
    C.fill_bank_torch(gu_dev[:n_gu], seed * 31 + 5, t, H)
    C.fill_bank_torch(dn_dev[:n_dn], seed * 31 + 6, t, I)
    return PrefillCase(OL.Geometry(H, I, E, K, t, t, glu), x, ids, w, sb, seed, gu_dev[:n_gu], dn_dev[:n_dn])


def prefill_oracle(case: PrefillCase, mode: int, tokens=None):
    """Oracle outputs (fp64 [T', H], bf16 bits, stages) for all tokens or a
    sample; only the experts those tokens route to are regenerated."""
    g = case.geom
    sel = np.arange(case.x.shape[0]) if tokens is None else np.asarray(tokens)
    routed = sorted({int(e) for e in case.ids[sel].reshape(-1) if 0 <= e < g.E})
    gu, dn = {}, {}
    for e in routed:
        gu[e] = C.bank_bytes_np(case.seed * 31 + 5, g.gate_up_type, g.H, e * 2 * g.I, 2 * g.I)
        dn[e] = C.bank_bytes_np(case.seed * 31 + 6, g.down_type, g.I, e * g.H, g.H)
    kind = {0: "nvfp4", 1: "q8_1", 2: "fp16", 3: "nvfp4"}[mode]   # 3: W4A4 arithmetic, fixed-order route sum
    return OL.moe_layer(g, gu, dn, case.sb, case.x[sel], case.ids[sel], case.w[sel], act_kind=kind, stages=True)


def run_prefill_gpu(case: PrefillCase, mode: int, stages=True):
    import torch

    from quantized_routed_expert_route_gb300 import capi
    g = case.geom
    T = case.x.shape[0]
    dev = "cuda"
    stream = torch.cuda.current_stream().cuda_stream
    sb = torch.from_numpy(case.sb).to(dev)
    geom = capi.moe_layer_geom(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, g.glu)
    bank = capi.moe_bank_create(geom, case.gu_dev.data_ptr(), case.gu_dev.numel(), case.dn_dev.data_ptr(),
                                case.dn_dev.numel(), sb.data_ptr(), capi.MOE_SRC_DEVICE_BORROW, stream)
    wsb = capi.moe_prefill_workspace_bytes(bank, T, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    x = torch.from_numpy(case.x.view(np.int16)).to(dev)
    ids = torch.from_numpy(case.ids).to(dev)
    w = torch.from_numpy(case.w).to(dev)
    out = torch.empty((T, g.H), dtype=torch.int16, device=dev)
    RT = T * g.top_k
    res = {}
    if stages:
        xq_bytes = {0: T * (g.H // 2 + g.H // 16), 1: T * (g.H // 32) * 36, 2: 2 * T * g.H,
                    3: T * (g.H // 2 + g.H // 16)}[mode]
        xq = torch.zeros(xq_bytes, dtype=torch.uint8, device=dev)
        off = torch.zeros(g.E + 1, dtype=torch.int32, device=dev)
        perm = torch.zeros(RT, dtype=torch.int32, device=dev)
        i16 = torch.zeros((RT, g.I), dtype=torch.float16, device=dev)
        capi.moe_debug_prefill_stages(bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), mode, out.data_ptr(),
                                      ws.data_ptr(), wsb, stream, xq.data_ptr(), off.data_ptr(), perm.data_ptr(),
                                      i16.data_ptr())
        torch.cuda.synchronize()
        res["xq"] = xq.cpu().numpy()
        res["off"] = off.cpu().numpy()
        res["perm"] = perm.cpu().numpy()
        res["i16"] = i16.cpu().numpy()
    else:
        capi.moe_prefill_grouped(bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), mode, out.data_ptr(),
                                 ws.data_ptr(), wsb, stream)
        torch.cuda.synchronize()
    res["out"] = out.cpu().numpy().view(np.uint16)
    res["err"] = capi.moe_get_error(ws.data_ptr(), wsb, stream)
    capi.moe_bank_destroy(bank)
    return res
