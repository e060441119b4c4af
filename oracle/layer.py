"""Oracle: one routed-expert MoE layer, decode and prompt path, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The layer formula is FreeToken PR #732, "Design":

    h = x @ W_gate_up^T;   g = h_gate * s_gate,  u = h_up * s_up
    y = (glu(g, u) @ W_down^T) * s_down * routing_weight         s per expert

with the [E,4] fp32 scale bank (s_gate, s_up, s_down, 1) of the same section.
The steps around it follow FreeToken PR #704, "How it plugs into the CPU
executor": prep_input (bf16 hidden -> the gate_up type's input, q8_1 for
quantized rows, float for BF16 rows), gate_up (a dot over every gate and up
row, then the activation), prep_inter (the intermediate -> the down type's
input), down (a dot over every output row, per route), and the executor's sum
over routes.  Strata PR #292, "Summary/Pipeline" fixes that each global scale
multiplies its own projection's fp32 output and is never folded.

The GLU is act(g) * u with act = SiLU, silu(g) = g / (1 + exp(-g)), or the
tanh form of GELU, gelu_tanh(g) = g/2 * (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
(Hendrycks and Gimpel, "Gaussian Error Linear Units", 2016); FreeToken PR
#732, "Other checks", runs experts with both.

Readings where the pages are silent:
  * gate rows are rows [0, I) of an expert's gate_up bank, up rows [I, 2I);
  * a route whose expert id is outside [0, E) contributes nothing;
  * the intermediate is cast to fp32 and quantized to q8_1 when the down
    type is quantized, and kept unquantized when it is BF16;
  * the output is the fp64 sum over routes rounded once to bf16 (ties even).

A quantized row dotted with a q8_1 activation equals, up to rounding order,
the dot of the dequantized row with the dequantized activation; this oracle
computes that plain definition with an fp64 matmul.

Pins (tests/test_oracle_layer.py): brute force over Python floats on the tiny
Q8_0 layer; with unit scales, one route and unit weight on a BF16 bank the
layer equals silu(x Wg^T) * (x Wu^T) Wd^T by numpy matmul; invariants
(linearity in the routing weight and in s_down, route-order independence,
invalid-id routes contribute zero).  Prompt-path W4A4 pins: see prefill().
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import formats as F


@dataclass
class Geometry:
    H: int
    I: int
    E: int
    top_k: int
    gate_up_type: int
    down_type: int
    glu: int = 0          # GLU_SILU or GLU_GELU_TANH


GLU_SILU, GLU_GELU_TANH = 0, 1


def silu(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def gelu_tanh(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore", invalid="ignore"):
        return 0.5 * g * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (g + 0.044715 * g ** 3)))


def _glu(g: np.ndarray, u: np.ndarray, kind: int) -> np.ndarray:
    if kind == GLU_SILU:
        return silu(g) * u
    if kind == GLU_GELU_TANH:
        return gelu_tanh(g) * u
    raise ValueError(kind)


class _ExpertCache:
    """Dequantizes an expert's rows once per call."""

    def __init__(self, geom: Geometry, gate_up, down):
        """gate_up / down: anything indexable by expert id that yields that
        expert's rows as uint8 ([2I, rb] and [H, rb]) -- a [E, rows, rb]
        array, or a mapping holding just the experts that are routed to."""
        self.g = geom
        self.rb_gu = F.row_bytes(geom.gate_up_type, geom.H)
        self.rb_d = F.row_bytes(geom.down_type, geom.I)
        self.gu, self.dn = gate_up, down
        self.cache: dict[int, tuple[np.ndarray, np.ndarray]] = {}

    def rows(self, e: int):
        if e not in self.cache:
            g = self.g
            gu = np.asarray(self.gu[e], dtype=np.uint8).reshape(2 * g.I, self.rb_gu)
            dn = np.asarray(self.dn[e], dtype=np.uint8).reshape(g.H, self.rb_d)
            self.cache[e] = (F.dequantize_rows(g.gate_up_type, gu, g.H),
                             F.dequantize_rows(g.down_type, dn, g.I))
        return self.cache[e]


def quantize_nvfp4_act(x32):
    """W4A4 activation quantizer of the prompt path (Strata PR #292,
    "Summary/Pipeline", W4A4): per 16 values, scale = UE4M3(amax/6) rounded
    to nearest-even with saturation (the global activation scale is 1, as
    FreeToken PR #732, "Design", leaves .input_scale unused), codes =
    E2M1(x / scale) rounded to nearest-even with saturation; an all-zero block
    has scale 0 and codes 0.  fp32 arithmetic throughout.

    Returns (codes uint8 [..., n], scales uint8 [..., n//16])."""
    x = np.asarray(x32, dtype=np.float32)
    xb = x.reshape(x.shape[:-1] + (x.shape[-1] // 16, 16))
    amax = np.max(np.abs(xb), axis=-1)
    sc = F.ue4m3_encode_rne_sat((amax / np.float32(6.0)).astype(np.float32))
    sv = F.ue4m3_value(sc).astype(np.float32)
    safe = np.where(sv > 0, sv, np.float32(1.0)).astype(np.float32)
    codes = F.e2m1_encode_rne_sat((xb / safe[..., None]).astype(np.float32))
    codes = np.where(sv[..., None] > 0, codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(x.shape), sc


def dequantize_nvfp4_act(codes, scales) -> np.ndarray:
    c = np.asarray(codes)
    v = F.e2m1_value(c).reshape(c.shape[:-1] + (c.shape[-1] // 16, 16))
    v = v * F.ue4m3_value(scales)[..., None]
    return v.reshape(c.shape)


def _act_in(kind: str, wtype: int, v32: np.ndarray) -> tuple[np.ndarray, dict]:
    """prep_input / prep_inter: fp32 values -> what the next dot consumes."""
    if wtype in F.FLOAT_TYPES:
        return v32.astype(np.float64), {}
    if kind == "q8_1":
        qs, d, s, sumq = F.quantize_q8_1(v32)
        return F.dequantize_q8_1(qs, d), {"qs": qs, "d": d, "s": s}
    if kind == "nvfp4":
        codes, scl = quantize_nvfp4_act(v32)
        return dequantize_nvfp4_act(codes, scl), {"codes": codes, "scales": scl}
    if kind == "fp16":
        # the FP16 prompt mode: no quantization, one IEEE rounding to fp16
        # (nearest even; beyond 65504 the value overflows to infinity)
        with np.errstate(over="ignore"):
            h = np.asarray(v32, dtype=np.float32).astype(np.float16)
        return h.astype(np.float64), {"f16": h}
    raise ValueError(kind)


def moe_layer(geom: Geometry, gate_up, down, scale_bank, x_bf16_bits, topk_ids, topk_w,
              act_kind: str = "q8_1", stages: bool = False):
    """Routed-expert layer for T tokens.

    x_bf16_bits: uint16 [T, H]; topk_ids: int [T, K]; topk_w: fp32 [T, K];
    scale_bank: fp32 [E, 4] or None (all ones); gate_up / down: the compact
    banks as uint8 arrays ([E, 2I, row_bytes] and [E, H, row_bytes]), or
    mappings from expert id to that expert's rows.
    act_kind: "q8_1" (decode and the W4A8 prompt path), "nvfp4" (W4A4) or
    "fp16" (the FP16 prompt mode: x and the fp32 intermediate rounded to fp16,
    not quantized; Strata PR #292, "Summary/Pipeline", lists W4A8, W4A4 and
    FP16 prompt modes).

    Returns (out_f64 [T, H], out_bf16_bits [T, H], stages dict or None)."""
    g = geom
    x = F.bf16_bits_to_f64(np.asarray(x_bf16_bits, dtype=np.uint16)).reshape(-1, g.H)
    T = x.shape[0]
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(T, g.top_k)
    w = np.asarray(topk_w, dtype=np.float32).reshape(T, g.top_k).astype(np.float64)
    if scale_bank is None:
        sb = np.ones((g.E, 4), dtype=np.float64)
    else:
        sb = np.asarray(scale_bank, dtype=np.float32).reshape(g.E, 4).astype(np.float64)
    cache = _ExpertCache(g, gate_up, down)
    out = np.zeros((T, g.H), dtype=np.float64)
    st = {"x_act": [], "x_hat": np.zeros((T, g.H)), "inter": np.zeros((T, g.top_k, g.I)),
          "inter_act": [], "inter_hat": np.zeros((T, g.top_k, g.I)),
          "y": np.zeros((T, g.top_k, g.H)), "valid": np.zeros((T, g.top_k), bool),
          "experts": cache.cache, "scales": sb, "w": w, "ids": ids} if stages else None
    for t in range(T):
        xa, xinfo = _act_in(act_kind, g.gate_up_type, x[t].astype(np.float32))
        if stages:
            st["x_act"].append(xinfo)
            st["x_hat"][t] = xa
        row_inter = []
        for k in range(g.top_k):
            e = int(ids[t, k])
            if not (0 <= e < g.E):
                row_inter.append(None)
                continue
            wgu, wd = cache.rows(e)
            h = wgu @ xa
            gg = h[: g.I] * sb[e, 0]
            uu = h[g.I:] * sb[e, 1]
            a = _glu(gg, uu, g.glu)
            aq, ainfo = _act_in(act_kind, g.down_type, a.astype(np.float32)
                                if g.down_type not in F.FLOAT_TYPES else a)
            if g.down_type in F.FLOAT_TYPES:
                aq = a
            y = (wd @ aq) * sb[e, 2] * w[t, k]
            out[t] += y
            if stages:
                st["inter"][t, k] = a
                st["inter_hat"][t, k] = aq
                st["y"][t, k] = y
                st["valid"][t, k] = True
            row_inter.append(ainfo)
        if stages:
            st["inter_act"].append(row_inter)
    out_bf16 = F.round_to_bf16(out)
    return out, F.f64_bf16_value_to_bits(out_bf16), st
