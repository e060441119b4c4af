"""Seeded inputs: hidden states, routings, scale banks and converted expert banks.

Recipes (the workload shapes of the layer configurations the pages describe):

  * hidden x ~ N(0, 1), rounded to bf16;
  * softmax routing: router logits ~ N(0, 1) [T, E], softmax, the top-k
    experts by probability (lower index first on ties), weights renormalised
    over the k chosen;
  * Zipf routing (the 47-layer stack): per layer a seeded permutation of the
    experts ranks them, log-popularity -s * log(rank), s = 1.1; each token
    takes the top-k of log-popularity plus Gumbel noise (k distinct experts),
    weights = softmax over the k chosen perturbed logits;
  * converted banks: fp32 weights ~ N(0, 0.02) written into the bank format
    the way an offline converter would (see each ``convert_*``).

Everything returns numpy arrays; bank rows are uint8 [rows, row_bytes].
"""
from __future__ import annotations

import numpy as np

BF16, Q8_0, Q4_K, NVFP4, Q6_K, Q4_0 = 0, 1, 2, 3, 4, 5
Q4_1, Q5_0, Q5_1, Q5_K, MXFP4 = 6, 7, 8, 9, 10
F16, F32 = 11, 12


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(wtype: int, k: int) -> int:
    return {BF16: 2 * k, Q8_0: k // 32 * 34, Q4_K: k // 256 * 144, NVFP4: k // 2 + k // 16,
            Q6_K: k // 256 * 210, Q4_0: k // 32 * 18, Q4_1: k // 32 * 20, Q5_0: k // 32 * 22,
            Q5_1: k // 32 * 24, Q5_K: k // 256 * 176, MXFP4: k // 32 * 17, F16: 2 * k, F32: 4 * k}[wtype]


# ------------------------------------------------------------------ activations / routing

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def hidden_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """x ~ N(0,1) as bf16 bits, uint16 [T, H]."""
    return f32_to_bf16_bits(rng(seed).standard_normal((T, H)).astype(np.float32))


def softmax_topk_routing(seed: int, T: int, E: int, k: int):
    """(ids int32 [T,k], weights fp32 [T,k]) from N(0,1) router logits."""
    logits = rng(seed).standard_normal((T, E))
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -p), axis=1)[:, :k]
    sel = np.take_along_axis(p, order, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def zipf_routing(seed: int, T: int, E: int, k: int, s: float = 1.1):
    """(ids int32 [T,k], weights fp32 [T,k]) with Zipf(s) expert popularity."""
    r = rng(seed)
    perm = r.permutation(E)
    logp = np.empty(E)
    logp[perm] = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    gumbel = -np.log(-np.log(r.random((T, E)).clip(1e-300, 1.0)))
    score = logp[None, :] + gumbel
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -score), axis=1)[:, :k]
    sel = np.take_along_axis(score, order, axis=1)
    w = np.exp(sel - sel.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


# ------------------------------------------------------------------ converters

def convert_bf16(w: np.ndarray) -> np.ndarray:
    """fp32 [R, K] -> bf16 rows (round to nearest even, by torch)."""
    return f32_to_bf16_bits(w).view(np.uint8).reshape(w.shape[0], 2 * w.shape[1])


def _e2m1_code(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code, saturating at 6) by counting
    the decision thresholds the magnitude passes; sign bit from the sign."""
    a = np.abs(v)
    mag = ((a > 0.25).astype(np.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
           + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    return (mag | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def convert_nvfp4(w: np.ndarray, s2: np.float32) -> np.ndarray:
    """ModelOpt-style NVFP4 rows from fp32 [R, K] with the projection's
    weight_scale_2 ``s2``: per 16 values the UE4M3 scale is
    e4m3((amax_blk / 6) / s2) (torch's float8_e4m3fn rounding, clamped at
    448), and each code is the nearest E2M1 of w / (scale * s2)."""
    import torch
    R, K = w.shape
    wb = w.astype(np.float32).reshape(R, K // 16, 16)
    amax = np.abs(wb).max(axis=-1)
    raw = np.minimum((amax / np.float32(6.0)).astype(np.float32) / np.float32(s2), np.float32(448.0))
    sc = torch.from_numpy(raw.astype(np.float32)).to(torch.float8_e4m3fn)
    sv = sc.to(torch.float32).numpy()
    scode = sc.view(torch.uint8).numpy().copy()
    den = (sv * np.float32(s2)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        x = np.where(den[..., None] > 0, wb / np.where(den > 0, den, 1)[..., None], 0).astype(np.float32)
    codes = _e2m1_code(x).reshape(R, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return np.concatenate([packed, scode.astype(np.uint8)], axis=1)


def _pack_q4k_scales(sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """Pack 8 six-bit (scale, min) pairs per super-block into 12 bytes (the
    inverse of the GGUF Q4_K unpack)."""
    out = np.zeros(sc.shape[:-1] + (12,), dtype=np.uint8)
    for j in range(4):
        out[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        out[..., j + 4] = (mn[..., j] & 63) | ((mn[..., j + 4] >> 4) << 6)
        out[..., j + 8] = (sc[..., j + 4] & 15) | ((mn[..., j + 4] & 15) << 4)
    return out


def convert_q4k(w: np.ndarray) -> np.ndarray:
    """Q4_K rows from fp32 [R, K] by a plain min/max encoder: per 32-value
    sub-block lo = min(0, min), step = (max - lo) / 15; per super-block
    d = max(step) / 63 and dmin = max(-lo) / 63 (fp16); 6-bit sc = round(step/d),
    m = round(-lo/dmin); codes = round((w + dmin*m) / (d*sc)) clipped to 0..15."""
    R, K = w.shape
    nsb = K // 256
    x = w.astype(np.float64).reshape(R, nsb, 8, 32)
    lo = np.minimum(0.0, x.min(axis=-1))
    hi = x.max(axis=-1)
    step = (hi - lo) / 15.0
    d = (step.max(axis=-1) / 63.0).astype(np.float16)
    dmin = ((-lo).max(axis=-1) / 63.0).astype(np.float16)
    d64, dmin64 = d.astype(np.float64), dmin.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d64[..., None] > 0, np.rint(step / d64[..., None]), 0).clip(0, 63).astype(np.int64)
        mn = np.where(dmin64[..., None] > 0, np.rint(-lo / dmin64[..., None]), 0).clip(0, 63).astype(np.int64)
        eff = d64[..., None] * sc
        q = np.where(eff[..., None] > 0,
                     np.rint((x + (dmin64[..., None] * mn)[..., None]) / np.where(eff > 0, eff, 1)[..., None]),
                     0).clip(0, 15).astype(np.uint8)
    out = np.zeros((R, nsb, 144), dtype=np.uint8)
    out[..., 0:2] = d.view(np.uint16)[..., None].view(np.uint8).reshape(R, nsb, 2)
    out[..., 2:4] = dmin.view(np.uint16)[..., None].view(np.uint8).reshape(R, nsb, 2)
    out[..., 4:16] = _pack_q4k_scales(sc, mn)
    qq = q.reshape(R, nsb, 4, 2, 32)                       # chunk c: sub-blocks 2c, 2c+1
    out[..., 16:144] = (qq[..., 0, :] | (qq[..., 1, :] << 4)).reshape(R, nsb, 128)
    return out.reshape(R, nsb * 144)


def convert_q6k(w: np.ndarray) -> np.ndarray:
    """Q6_K rows from fp32 [R, K] by a plain absmax encoder: per 16 values
    step = amax / 31; per super-block d = max(step) / 127 (fp16); int8 scale
    round(step / d); codes round(w / (d * scale)) + 32 clipped to 0..63, packed
    into ql (low 4 bits) and qh (high 2 bits) in the GGUF order (value
    128n + 32c + l: nibble c // 2 of ql[64n + 32(c % 2) + l], bits 2c..2c+1 of
    qh[32n + l])."""
    R, K = w.shape
    nsb = K // 256
    x = w.astype(np.float64).reshape(R, nsb, 16, 16)
    step = np.abs(x).max(axis=-1) / 31.0
    d = (step.max(axis=-1) / 127.0).astype(np.float16)
    d64 = d.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d64[..., None] > 0, np.rint(step / d64[..., None]), 0).clip(-128, 127).astype(np.int64)
        eff = d64[..., None] * sc
        q = np.where(eff[..., None] != 0, np.rint(x / np.where(eff != 0, eff, 1)[..., None]), 0)
    q = (q + 32).clip(0, 63).astype(np.int64).reshape(R, nsb, 256)
    out = np.zeros((R, nsb, 210), dtype=np.uint8)
    for n in range(2):
        for c in range(4):
            v = q[..., 128 * n + 32 * c: 128 * n + 32 * c + 32]
            lo, hi = v & 0x0F, v >> 4
            o = 64 * n + 32 * (c % 2)
            out[..., o: o + 32] |= (lo << (4 * (c // 2))).astype(np.uint8)
            out[..., 128 + 32 * n: 128 + 32 * n + 32] |= (hi << (2 * c)).astype(np.uint8)
    out[..., 192:208] = sc.astype(np.int8).view(np.uint8)
    out[..., 208:210] = d.view(np.uint16)[..., None].view(np.uint8).reshape(R, nsb, 2)
    return out.reshape(R, nsb * 210)


def convert_q4_0(w: np.ndarray) -> np.ndarray:
    """Q4_0 rows from fp32 [R, K]: per 32 values d = amax / 7 (fp16), codes
    round(w / d) + 8 clipped to 0..15; value j < 16 in the low nibble of code
    byte j, value j + 16 in its high nibble."""
    R, K = w.shape
    nb = K // 32
    x = w.astype(np.float64).reshape(R, nb, 32)
    d = (np.abs(x).max(axis=-1) / 7.0).astype(np.float16)
    d64 = d.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d64[..., None] > 0, np.rint(x / np.where(d64 > 0, d64, 1)[..., None]), 0)
    q = (q + 8).clip(0, 15).astype(np.uint8)
    out = np.zeros((R, nb, 18), dtype=np.uint8)
    out[..., 0:2] = d.view(np.uint16)[..., None].view(np.uint8).reshape(R, nb, 2)
    out[..., 2:18] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(R, nb * 18)


def _f16_bytes(v: np.ndarray) -> np.ndarray:
    """fp16 values [...] -> their two little-endian bytes [..., 2]."""
    return v.astype(np.float16).view(np.uint16)[..., None].view(np.uint8).reshape(v.shape + (2,))


def _nibble_split(q: np.ndarray) -> np.ndarray:
    """32 codes (0..15) per block -> 16 bytes: value j low nibble, j+16 high."""
    return (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8)


def _q5_high_word(q: np.ndarray) -> np.ndarray:
    """The fifth bits of 32 5-bit codes as 4 little-endian bytes (bit j: value j)."""
    bits = ((q >> 4) & 1).astype(np.uint64)
    word = (bits << np.arange(32, dtype=np.uint64)).sum(axis=-1).astype(np.uint32)
    return word[..., None].view(np.uint8).reshape(q.shape[:-1] + (4,))


def convert_q4_1_q5(w: np.ndarray, wtype: int) -> np.ndarray:
    """Q4_1 / Q5_0 / Q5_1 rows from fp32 [R, K], per 32 values.  Q4_1 and
    Q5_1 (value d*q + m): m = fp16(min), d = fp16((max - min) / (2^bits - 1)),
    q = round((w - m) / d) clipped.  Q5_0 (value d*(q - 16)): d = fp16(amax /
    15), q = round(w / d) + 16 clipped to 0..31."""
    R, K = w.shape
    x = w.astype(np.float64).reshape(R, K // 32, 32)
    with np.errstate(divide="ignore", invalid="ignore"):
        if wtype == Q5_0:
            d = (np.abs(x).max(axis=-1) / 15.0).astype(np.float16)
            d64 = d.astype(np.float64)
            q = (np.where(d64[..., None] > 0, np.rint(x / np.where(d64 > 0, d64, 1)[..., None]), 0) + 16).clip(0, 31)
            m = None
        else:
            top = 15.0 if wtype == Q4_1 else 31.0
            m = x.min(axis=-1).astype(np.float16)
            d = ((x.max(axis=-1) - m.astype(np.float64)) / top).astype(np.float16)
            d64 = d.astype(np.float64)
            q = np.where(d64[..., None] > 0,
                         np.rint((x - m.astype(np.float64)[..., None]) / np.where(d64 > 0, d64, 1)[..., None]),
                         0).clip(0, top)
    q = q.astype(np.int64)
    parts = [_f16_bytes(d)]
    if m is not None:
        parts.append(_f16_bytes(m))
    if wtype != Q4_1:
        parts.append(_q5_high_word(q))
    parts.append(_nibble_split(q & 15))
    return np.concatenate(parts, axis=-1).reshape(R, -1)


def convert_q5k(w: np.ndarray) -> np.ndarray:
    """Q5_K rows from fp32 [R, K]: the Q4_K min/max encoder with 5-bit codes
    (step = (max - lo) / 31), the low 4 bits laid out as Q4_K, the fifth bit
    of value l of sub-block j in bit j of high-bit byte l."""
    R, K = w.shape
    nsb = K // 256
    x = w.astype(np.float64).reshape(R, nsb, 8, 32)
    lo = np.minimum(0.0, x.min(axis=-1))
    step = (x.max(axis=-1) - lo) / 31.0
    d = (step.max(axis=-1) / 63.0).astype(np.float16)
    dmin = ((-lo).max(axis=-1) / 63.0).astype(np.float16)
    d64, dmin64 = d.astype(np.float64), dmin.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d64[..., None] > 0, np.rint(step / d64[..., None]), 0).clip(0, 63).astype(np.int64)
        mn = np.where(dmin64[..., None] > 0, np.rint(-lo / dmin64[..., None]), 0).clip(0, 63).astype(np.int64)
        eff = d64[..., None] * sc
        q = np.where(eff[..., None] > 0,
                     np.rint((x + (dmin64[..., None] * mn)[..., None]) / np.where(eff > 0, eff, 1)[..., None]),
                     0).clip(0, 31).astype(np.int64)
    out = np.zeros((R, nsb, 176), dtype=np.uint8)
    out[..., 0:2] = _f16_bytes(d)
    out[..., 2:4] = _f16_bytes(dmin)
    out[..., 4:16] = _pack_q4k_scales(sc, mn)
    hb = ((q >> 4) & 1).astype(np.uint8)                  # [R, nsb, 8, 32]
    out[..., 16:48] = (hb << np.arange(8, dtype=np.uint8)[:, None]).sum(axis=-2).astype(np.uint8)
    qq = (q & 15).astype(np.uint8).reshape(R, nsb, 4, 2, 32)
    out[..., 48:176] = (qq[..., 0, :] | (qq[..., 1, :] << 4)).reshape(R, nsb, 128)
    return out.reshape(R, nsb * 176)


def convert_mxfp4(w: np.ndarray) -> np.ndarray:
    """MXFP4 rows from fp32 [R, K]: per 32 values the E8M0 exponent e =
    127 + ceil(log2(amax / 6)) (so amax / 2^(e-127) <= 6), codes the nearest
    E2M1 of w / 2^(e-127)."""
    R, K = w.shape
    x = w.astype(np.float64).reshape(R, K // 32, 32)
    amax = np.abs(x).max(axis=-1)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1) / 6.0)), -127)
    e = np.clip(ex + 127, 0, 254).astype(np.int64)
    codes = _e2m1_code(x / np.ldexp(1.0, e - 127)[..., None]).astype(np.int64)
    out = np.concatenate([e.astype(np.uint8)[..., None], _nibble_split(codes)], axis=-1)
    return out.reshape(R, -1)


def convert_float(w: np.ndarray, wtype: int) -> np.ndarray:
    """F16 rows (round to nearest even) or F32 rows from fp32 [R, K]."""
    v = w.astype(np.float16) if wtype == F16 else w.astype(np.float32)
    return np.ascontiguousarray(v).view(np.uint8).reshape(w.shape[0], -1)


def q8_0_codes_bank(seed: int, rows: int, k: int) -> np.ndarray:
    """Q8_0 rows with int8 codes uniform in [-127, 127] and fp16 scales
    uniform in (1e-4, 5e-4) (the tiny single-layer configuration)."""
    r = rng(seed)
    nb = k // 32
    q = r.integers(-127, 128, size=(rows, nb, 32)).astype(np.int8)
    d = r.uniform(1e-4, 5e-4, size=(rows, nb)).astype(np.float16)
    out = np.zeros((rows, nb, 34), dtype=np.uint8)
    out[..., 0:2] = d.view(np.uint16)[..., None].view(np.uint8).reshape(rows, nb, 2)
    out[..., 2:34] = q.view(np.uint8)
    return out.reshape(rows, nb * 34)


def converted_expert(seed: int, e: int, H: int, I: int, gate_up_type: int, down_type: int):
    """One converted expert: (gate_up uint8 [2I, rb_gu], down uint8 [H, rb_d],
    scales fp32 [4]).  Weights ~ N(0, 0.02) (Q8_0: the direct code recipe);
    NVFP4 projections get s2 = amax / (6 * 448) each (gate, up, down)."""
    r = rng(seed * 100003 + e)
    sc = np.ones(4, dtype=np.float32)
    if gate_up_type == Q8_0:
        gu = q8_0_codes_bank(seed * 100003 + e, 2 * I, H)
    else:
        wg = (r.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
        if gate_up_type == NVFP4:
            parts = []
            for p, (a, b) in enumerate(((0, I), (I, 2 * I))):
                s2 = np.float32(np.abs(wg[a:b]).max() / np.float32(6.0 * 448.0))
                sc[p] = s2
                parts.append(convert_nvfp4(wg[a:b], s2))
            gu = np.concatenate(parts, axis=0)
        elif gate_up_type == Q4_K:
            gu = convert_q4k(wg)
        elif gate_up_type == Q6_K:
            gu = convert_q6k(wg)
        elif gate_up_type == Q4_0:
            gu = convert_q4_0(wg)
        elif gate_up_type in (Q4_1, Q5_0, Q5_1):
            gu = convert_q4_1_q5(wg, gate_up_type)
        elif gate_up_type == Q5_K:
            gu = convert_q5k(wg)
        elif gate_up_type == MXFP4:
            gu = convert_mxfp4(wg)
        elif gate_up_type in (F16, F32):
            gu = convert_float(wg, gate_up_type)
        else:
            gu = convert_bf16(wg)
    if down_type == Q8_0:
        dn = q8_0_codes_bank(seed * 100003 + e + 50000, H, I)
    else:
        wd = (r.standard_normal((H, I)) * 0.02).astype(np.float32)
        if down_type == NVFP4:
            s2 = np.float32(np.abs(wd).max() / np.float32(6.0 * 448.0))
            sc[2] = s2
            dn = convert_nvfp4(wd, s2)
        elif down_type == Q4_K:
            dn = convert_q4k(wd)
        elif down_type == Q6_K:
            dn = convert_q6k(wd)
        elif down_type == Q4_0:
            dn = convert_q4_0(wd)
        elif down_type in (Q4_1, Q5_0, Q5_1):
            dn = convert_q4_1_q5(wd, down_type)
        elif down_type == Q5_K:
            dn = convert_q5k(wd)
        elif down_type == MXFP4:
            dn = convert_mxfp4(wd)
        elif down_type in (F16, F32):
            dn = convert_float(wd, down_type)
        else:
            dn = convert_bf16(wd)
    return gu, dn, sc


def converted_layer(seed: int, H: int, I: int, E: int, gate_up_type: int, down_type: int,
                    experts=None, filler_seed: int | None = None):
    """A converted layer: (gate_up uint8 [E, 2I, rb_gu], down uint8 [E, H, rb_d],
    scale bank fp32 [E, 4]).

    Weights ~ N(0, 0.02).  Q8_0 banks use the direct code recipe instead.
    NVFP4 projections get s2 = amax / (6 * 448) per expert per projection
    (gate, up and down separately); other types get scale 1.  The fourth
    column of the scale bank is 1.

    ``experts``: if given, only these experts are converted; the others are
    filled from the counter-based generator (``filler_seed``), which is much
    faster for full-size layers where only the routed experts are read."""
    from . import counter
    rb_gu, rb_d = row_bytes(gate_up_type, H), row_bytes(down_type, I)
    gu = np.empty((E, 2 * I, rb_gu), dtype=np.uint8)
    dn = np.empty((E, H, rb_d), dtype=np.uint8)
    sb = np.ones((E, 4), dtype=np.float32)
    todo = range(E) if experts is None else sorted(set(int(e) for e in experts))
    if experts is not None:
        fs = seed * 7919 + 17 if filler_seed is None else filler_seed
        gu[:] = counter.bank_bytes_np(fs, gate_up_type, H, 0, E * 2 * I).reshape(E, 2 * I, rb_gu)
        dn[:] = counter.bank_bytes_np(fs + 1, down_type, I, 0, E * H).reshape(E, H, rb_d)
    for e in todo:
        gu[e], dn[e], sb[e] = converted_expert(seed, e, H, I, gate_up_type, down_type)
    return gu, dn, sb


def counter_scale_bank(seed: int, E: int, gate_up_type: int, down_type: int) -> np.ndarray:
    """Scale bank for counter-based banks: NVFP4 projections get a
    weight_scale_2 in [0.004, 0.006), other types 1; fourth column 1."""
    r = rng(seed)
    sb = np.ones((E, 4), dtype=np.float32)
    v = r.uniform(0.004, 0.006, size=(E, 3)).astype(np.float32)
    if gate_up_type == NVFP4:
        sb[:, 0:2] = v[:, 0:2]
    if down_type == NVFP4:
        sb[:, 2] = v[:, 2]
    return sb
