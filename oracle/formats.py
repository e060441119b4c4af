"""Oracle: the block formats of the expert banks and activations, as plain numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Formats and where they come from:

  * q8_1 activation block -- 32 int8 codes, an fp16 scale d and an fp16 sum
    s.  The q8_1 input quantizer is named in FreeToken PR #704 ("How it plugs
    into the CPU executor", prep_input) and Strata PR #292 ("Summary/Pipeline",
    Decode: "q8_1 activations").  The pages print no formula; the reading used
    here is: d = amax/127 in fp32 (IEEE division), q = round-half-even(x/d) in
    fp32 (0 when d = 0), stored d_h = fp16(d), s_h = fp16(d * sum(q)) with the
    product taken in fp32.
  * Q8_0 weight block -- fp16 d then 32 int8 codes (34 bytes), value d*q.
  * Q4_K super-block -- 256 values in 144 bytes: fp16 d, fp16 dmin, 12 bytes
    of packed 6-bit (scale, min) pairs for 8 sub-blocks of 32, 128 bytes of
    4-bit codes; value d*sc_j*q - dmin*m_j.  Sizes from FreeToken issue #194,
    "Reproduction geometry"; the bit layout is the public GGUF one (the pages
    give only byte counts).
  * NVFP4 -- E2M1 codes with one UE4M3 scale per 16 values ("group 16",
    Strata PR #292, "Summary/Pipeline") and a per-expert fp32 weight_scale_2
    applied to the projection output (FreeToken PR #732, "Design").  Row
    layout of this library (the pages fix none): the K/2 code bytes (element
    2i in the low nibble of byte i, 2i+1 in the high nibble) followed by the
    K/16 scale bytes.
  * BF16 rows -- raw little-endian bf16 (FreeToken issue #194, "Proposed
    design": BF16 rows go to a dense kernel, not MMVQ).  F16 and F32 rows
    (raw little-endian fp16 / fp32) are the other float rows of FreeToken PR
    #704's synthetic list ("Validation": F16, F32, BF16 with quantized
    partners); like BF16 they keep the activations float.
  * Q6_K super-block -- 256 values in 210 bytes: ql[128] (low 4 bits of each
    code), qh[64] (high 2 bits), scales[16] (int8, one per 16 values), fp16
    d; value d*scale_g*(q - 32) with q the 6-bit code.  Q4_0 block -- fp16 d
    then 16 bytes of 4-bit codes, value d*(q - 8).  Both are among the GGUF
    types of FreeToken PR #704 ("Tests": the Q4_0 rows of the real Gemma
    checkpoint, and Q6_K in the synthetic type list); the bit layouts are the
    public GGUF ones, stated in prose at q6k_codes and q4_0_codes (the pages
    give neither), so GGUF byte compatibility is unpinned.
  * Q4_1, Q5_0, Q5_1, Q5_K and MXFP4 -- the remaining types of the synthetic
    list in FreeToken PR #704 ("Validation": Q4_1, Q5_1, Q4_K, Q5_0, Q6_K,
    MXFP4, Q5_K rows).  32-value blocks: Q4_1 fp16 d, fp16 m, 16 code bytes,
    value d*q + m; Q5_0 fp16 d, a 32-bit word of high bits, 16 code bytes,
    value d*(q - 16); Q5_1 fp16 d, fp16 m, the high-bit word, 16 code
    bytes, value d*q + m; MXFP4 one E8M0 byte e then 16 code bytes of E2M1,
    value E2M1(code) * 2^(e - 127).  Q5_K: 256 values in 176 bytes, the Q4_K
    header (d, dmin, 12 packed scale bytes), 32 bytes of high bits, 128 code
    bytes; value d*sc_j*q - dmin*m_j with 5-bit q.  Public GGUF layouts,
    stated in prose at each decoder; GGUF byte compatibility is unpinned.

Pins (tests/test_oracle_formats.py): UE4M3 against torch's float8_e4m3fn
decoder over all 127 finite codes; E2M1 against the same decoder through the
E2M1-in-E4M3 embedding; fp16/bf16 via numpy bit views; Q4_K unpack by an
exhaustive single-bit invariant plus a hand-worked golden super-block; Q6_K and
Q4_0 codes by the same single-bit invariant and hand-worked values; q8_1 by
crafted vectors with hand-computed results and the round-trip bound; integer
block dots by brute force over Python ints.
"""
from __future__ import annotations

import numpy as np

QK8 = 32          # q8_1 / Q8_0 block length
QK_K = 256        # Q4_K super-block length
NVFP4_GROUP = 16  # values per UE4M3 scale

TYPE_BF16, TYPE_Q8_0, TYPE_Q4_K, TYPE_NVFP4, TYPE_Q6_K, TYPE_Q4_0 = 0, 1, 2, 3, 4, 5
TYPE_Q4_1, TYPE_Q5_0, TYPE_Q5_1, TYPE_Q5_K, TYPE_MXFP4 = 6, 7, 8, 9, 10
TYPE_F16, TYPE_F32 = 11, 12
TYPE_NAMES = {TYPE_BF16: "bf16", TYPE_Q8_0: "q8_0", TYPE_Q4_K: "q4_k", TYPE_NVFP4: "nvfp4", TYPE_Q6_K: "q6_k",
              TYPE_Q4_0: "q4_0", TYPE_Q4_1: "q4_1", TYPE_Q5_0: "q5_0", TYPE_Q5_1: "q5_1", TYPE_Q5_K: "q5_k",
              TYPE_MXFP4: "mxfp4", TYPE_F16: "f16", TYPE_F32: "f32"}
# float rows: the activations stay float (no q8_1), the intermediate stays fp32
FLOAT_TYPES = (TYPE_BF16, TYPE_F16, TYPE_F32)

Q8_1_BLOCK_BYTES = 36   # fp16 d, fp16 s, 32 int8


def row_bytes(wtype: int, k: int) -> int:
    """Bytes of one bank row of ``k`` values; 0 when ``k`` is not a whole
    number of blocks.  FreeToken PR #704, "How it plugs into the CPU executor"
    (each bank holds rows of row_bytes(type, K))."""
    if wtype in (TYPE_BF16, TYPE_F16):
        return 2 * k if k % 32 == 0 else 0
    if wtype == TYPE_F32:
        return 4 * k if k % 32 == 0 else 0
    if wtype == TYPE_Q8_0:
        return (k // 32) * 34 if k % 32 == 0 else 0
    if wtype == TYPE_Q4_K:
        return (k // 256) * 144 if k % 256 == 0 else 0
    if wtype == TYPE_NVFP4:
        return k // 2 + k // 16 if k % 32 == 0 else 0
    if wtype == TYPE_Q6_K:
        return (k // 256) * 210 if k % 256 == 0 else 0
    if wtype == TYPE_Q4_0:
        return (k // 32) * 18 if k % 32 == 0 else 0
    per32 = {TYPE_Q4_1: 20, TYPE_Q5_0: 22, TYPE_Q5_1: 24, TYPE_MXFP4: 17}
    if wtype in per32:
        return (k // 32) * per32[wtype] if k % 32 == 0 else 0
    if wtype == TYPE_Q5_K:
        return (k // 256) * 176 if k % 256 == 0 else 0
    return 0


# ---------------------------------------------------------------- scalar codecs

def fp16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), once.

    bf16 keeps 8 significant bits and fp32's exponent range; below 2^-126 the
    spacing is the subnormal quantum 2^-133.  Returns fp64 values that are
    exactly representable in bf16 (overflow -> +-inf)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    _, ex = np.frexp(x[nz])                     # |x| in [2^(ex-1), 2^ex)
    q = np.exp2(np.maximum(ex.astype(np.float64) - 8.0, -133.0))
    r = np.rint(x[nz] / q) * q
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def f64_bf16_value_to_bits(v) -> np.ndarray:
    """Bits of values that are already exact bf16 numbers."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e2m1_value(code) -> np.ndarray:
    """E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
    Exponent 0 is subnormal: m * 0.5.  Magnitudes {0,.5,1,1.5,2,3,4,6}."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e.astype(np.float64) - 1.0))
    return sign * mag


def ue4m3_value(byte) -> np.ndarray:
    """UE4M3 (unsigned E4M3, bias 7): bits 6..3 exponent, 2..0 mantissa.
    Exponent 0 is subnormal m * 2^-9; 0x7F is NaN; bit 7 set is not a valid
    unsigned code and also decodes to NaN."""
    b = np.asarray(byte, dtype=np.int64)
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where(((b & 0x7F) == 0x7F) | ((b & 0x80) != 0), np.nan, val)
    return val


_E2M1_MAGS = e2m1_value(np.arange(8))           # codes 0..7
_UE4M3_FINITE = ue4m3_value(np.arange(0x7F))    # codes 0..0x7E


def _nearest_code_ties_even(v, table) -> np.ndarray:
    """Index of the nearest entry of the ascending ``table`` to each |v|;
    ties go to the even index (the even code).  Values above the last entry
    saturate to it."""
    a = np.asarray(v, dtype=np.float64)
    hi = np.searchsorted(table, a, side="left")
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    dlo = np.abs(a - table[lo])
    dhi = np.abs(table[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return pick.astype(np.int64)


def ue4m3_encode_rne_sat(v32) -> np.ndarray:
    """fp32 value >= 0 -> UE4M3 code, round to nearest with ties to even,
    saturating at 0x7E (448).  Prompt path, Strata PR #292, "Summary/
    Pipeline" (W4A4: activations quantized to NVFP4 on the fly)."""
    a = np.asarray(v32, dtype=np.float32).astype(np.float64)
    return _nearest_code_ties_even(a, _UE4M3_FINITE).astype(np.uint8)


def e2m1_encode_rne_sat(v32) -> np.ndarray:
    """fp32 value -> E2M1 code, nearest magnitude with ties to the even code,
    saturating at 6; the sign bit follows the sign of the input (a negative
    value that rounds to zero gives code 8, i.e. -0)."""
    a = np.asarray(v32, dtype=np.float32).astype(np.float64)
    mag = _nearest_code_ties_even(np.abs(a), _E2M1_MAGS)
    return (mag | np.where(np.signbit(a), 8, 0)).astype(np.uint8)


# ---------------------------------------------------------------- q8_1

def quantize_q8_1(x32):
    """Quantize fp32 values (last axis a multiple of 32) to q8_1 blocks.

    Returns (qs int8 [..., nb, 32], d_h fp16 bits [..., nb], s_h fp16 bits
    [..., nb], sumq int64 [..., nb]).  Every step is in fp32, as the reading
    in the module docstring states."""
    x = np.asarray(x32, dtype=np.float32)
    assert x.shape[-1] % QK8 == 0
    xb = x.reshape(x.shape[:-1] + (x.shape[-1] // QK8, QK8))
    amax = np.max(np.abs(xb), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    q = np.rint((xb / safe[..., None]).astype(np.float32))
    q = np.where(d[..., None] > 0, q, np.float32(0.0))
    qs = q.astype(np.int8)
    sumq = qs.astype(np.int64).sum(axis=-1)
    d_h = d.astype(np.float16)
    s_h = (d * sumq.astype(np.float32)).astype(np.float32).astype(np.float16)
    return qs, d_h.view(np.uint16), s_h.view(np.uint16), sumq


def dequantize_q8_1(qs, d_bits) -> np.ndarray:
    """q * fp16(d) in fp64, flattened back to [..., nb*32]."""
    v = np.asarray(qs, dtype=np.float64) * fp16_bits_to_f64(d_bits)[..., None]
    return v.reshape(v.shape[:-2] + (v.shape[-2] * v.shape[-1],))


def q8_1_pack_blocks(qs, d_bits, s_bits) -> np.ndarray:
    """Serialise q8_1 blocks into the 36-byte block format (d, s, qs[32])."""
    nb = qs.shape[-2]
    lead = qs.shape[:-2]
    out = np.zeros(lead + (nb, Q8_1_BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = np.asarray(d_bits, dtype=np.uint16)[..., None].view(np.uint8).reshape(lead + (nb, 2))
    out[..., 2:4] = np.asarray(s_bits, dtype=np.uint16)[..., None].view(np.uint8).reshape(lead + (nb, 2))
    out[..., 4:36] = np.asarray(qs, dtype=np.int8).view(np.uint8)
    return out


# ---------------------------------------------------------------- weight rows

def q4k_scale_min(scales12) -> tuple[np.ndarray, np.ndarray]:
    """Unpack the 12 packed bytes of a Q4_K super-block into 8 (sc, m) pairs
    of 6 bits.  Sub-blocks 0..3: low 6 bits of bytes j (sc) and j+4 (m).
    Sub-blocks 4..7: low nibble (sc) / high nibble (m) of byte j+4, with the
    top two bits taken from the top two bits of byte j-4 (sc) / byte j (m)."""
    s = np.asarray(scales12, dtype=np.int64)
    sc = np.zeros(s.shape[:-1] + (8,), dtype=np.int64)
    mn = np.zeros_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        mn[..., j] = s[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (s[..., j + 4] & 0x0F) | ((s[..., j - 4] >> 6) << 4)
        mn[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, mn


def q4k_codes(qs128) -> np.ndarray:
    """The 256 4-bit codes of a super-block in value order.  Byte l of chunk c
    (32 bytes each) holds sub-block 2c value l in its low nibble and sub-block
    2c+1 value l in its high nibble."""
    q = np.asarray(qs128, dtype=np.int64)
    q = q.reshape(q.shape[:-1] + (4, 32))
    lo = q & 0x0F
    hi = q >> 4
    out = np.stack([lo, hi], axis=-2)            # [..., 4 chunks, 2, 32]
    return out.reshape(out.shape[:-3] + (256,))


def q6k_codes(sb210) -> np.ndarray:
    """The 256 signed codes q - 32 (in [-32, 31]) of Q6_K super-blocks
    (uint8 [..., 210]) in value order.  Value v = 128*n + 32*c + l (half n,
    quarter c, lane l < 32): its low 4 bits are nibble c // 2 (low nibble
    first) of ql byte 64*n + 32*(c % 2) + l, its high 2 bits are bits 2c and
    2c+1 of qh byte 32*n + l."""
    b = np.asarray(sb210, dtype=np.int64)
    ql, qh = b[..., 0:128], b[..., 128:192]
    out = np.zeros(b.shape[:-1] + (256,), dtype=np.int64)
    for n in range(2):
        for c in range(4):
            lo = (ql[..., 64 * n + 32 * (c % 2): 64 * n + 32 * (c % 2) + 32] >> (4 * (c // 2))) & 0x0F
            hi = (qh[..., 32 * n: 32 * n + 32] >> (2 * c)) & 3
            out[..., 128 * n + 32 * c: 128 * n + 32 * c + 32] = (lo | (hi << 4)) - 32
    return out


def q6k_scales(sb210) -> np.ndarray:
    """The 16 signed 8-bit scales of Q6_K super-blocks; scale g covers values
    16g .. 16g+15."""
    return np.asarray(sb210, dtype=np.uint8)[..., 192:208].view(np.int8).astype(np.int64)


def q4_0_codes(blk18) -> np.ndarray:
    """The 32 signed codes q - 8 (in [-8, 7]) of Q4_0 blocks (uint8 [..., 18])
    in value order: value j < 16 is the low nibble of code byte j, value j+16
    its high nibble."""
    b = np.asarray(blk18, dtype=np.int64)[..., 2:18]
    return np.concatenate([b & 0x0F, b >> 4], axis=-1) - 8


def nibble_split_codes(qs16) -> np.ndarray:
    """The 32 4-bit codes of a block's 16 code bytes in value order: value j
    < 16 is the low nibble of byte j, value j + 16 its high nibble (Q4_0,
    Q4_1, Q5_0, Q5_1, MXFP4)."""
    b = np.asarray(qs16, dtype=np.int64)
    return np.concatenate([b & 0x0F, b >> 4], axis=-1)


def q5_high_bits(qh4) -> np.ndarray:
    """The 32 high bits of a Q5_0 / Q5_1 block: bit j of the little-endian
    32-bit word qh is the fifth bit (value 16) of value j's code."""
    b = np.asarray(qh4, dtype=np.int64)
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    return (word[..., None] >> np.arange(32)) & 1


def q5k_codes(sb176) -> np.ndarray:
    """The 256 5-bit codes of Q5_K super-blocks in value order: the low 4
    bits as in Q4_K (code byte l of chunk c: sub-block 2c in the low nibble,
    2c+1 in the high nibble), the fifth bit of value l of sub-block j is bit
    j of high-bit byte l."""
    b = np.asarray(sb176, dtype=np.int64)
    lo = q4k_codes(b[..., 48:176]).reshape(b.shape[:-1] + (8, 32))
    qh = b[..., 16:48]                                        # [..., 32]
    hi = (qh[..., None, :] >> np.arange(8)[:, None]) & 1      # [..., 8 sub-blocks, 32]
    return (lo | (hi << 4)).reshape(b.shape[:-1] + (256,))


def e8m0_value(e) -> np.ndarray:
    """E8M0 (the MXFP4 block scale): 2^(e - 127) for e = 0..254; 255 is not a
    finite scale (NaN in the microscaling formats) and is kept out of banks."""
    e = np.asarray(e, dtype=np.int64)
    assert (e < 255).all()
    return np.ldexp(1.0, e - 127)


def dequantize_rows(wtype: int, rows, k: int) -> np.ndarray:
    """Decode bank rows (uint8 [R, row_bytes(wtype, k)]) to fp64 [R, k].

    The per-expert weight_scale_2 is NOT applied here: FreeToken PR #732,
    "Design", applies it to the matmul result of each projection."""
    rows = np.asarray(rows, dtype=np.uint8)
    rb = row_bytes(wtype, k)
    assert rb > 0 and rows.shape[-1] == rb, (wtype, k, rows.shape)
    r = rows.shape[0]
    if wtype == TYPE_BF16:
        return bf16_bits_to_f64(rows.view(np.uint16)).reshape(r, k)
    if wtype == TYPE_F16:
        return fp16_bits_to_f64(rows.view(np.uint16)).reshape(r, k)
    if wtype == TYPE_F32:
        return rows.view("<f4").astype(np.float64).reshape(r, k)
    if wtype == TYPE_Q8_0:
        blk = rows.reshape(r, k // 32, 34)
        d = fp16_bits_to_f64(blk[..., 0:2].copy().view(np.uint16)[..., 0])
        q = blk[..., 2:34].view(np.int8).astype(np.float64)
        return (q * d[..., None]).reshape(r, k)
    if wtype == TYPE_Q4_K:
        sb = rows.reshape(r, k // 256, 144)
        d = fp16_bits_to_f64(sb[..., 0:2].copy().view(np.uint16)[..., 0])
        dmin = fp16_bits_to_f64(sb[..., 2:4].copy().view(np.uint16)[..., 0])
        sc, mn = q4k_scale_min(sb[..., 4:16])
        q = q4k_codes(sb[..., 16:144]).reshape(r, k // 256, 8, 32).astype(np.float64)
        v = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None]
        return v.reshape(r, k)
    if wtype == TYPE_NVFP4:
        codes = rows[:, : k // 2].astype(np.int64)
        scl = rows[:, k // 2: k // 2 + k // 16]
        nib = np.stack([codes & 0x0F, codes >> 4], axis=-1).reshape(r, k)
        v = e2m1_value(nib) * np.repeat(ue4m3_value(scl), NVFP4_GROUP, axis=-1)
        return v
    if wtype == TYPE_Q6_K:
        sb = rows.reshape(r, k // 256, 210)
        d = fp16_bits_to_f64(sb[..., 208:210].copy().view(np.uint16)[..., 0])
        q = q6k_codes(sb).reshape(r, k // 256, 16, 16).astype(np.float64)
        v = d[..., None, None] * q6k_scales(sb)[..., None] * q
        return v.reshape(r, k)
    if wtype == TYPE_Q4_0:
        blk = rows.reshape(r, k // 32, 18)
        d = fp16_bits_to_f64(blk[..., 0:2].copy().view(np.uint16)[..., 0])
        return (q4_0_codes(blk) * d[..., None]).reshape(r, k)
    if wtype in (TYPE_Q4_1, TYPE_Q5_0, TYPE_Q5_1):
        nbytes = {TYPE_Q4_1: 20, TYPE_Q5_0: 22, TYPE_Q5_1: 24}[wtype]
        blk = rows.reshape(r, k // 32, nbytes)
        d = fp16_bits_to_f64(blk[..., 0:2].copy().view(np.uint16)[..., 0])
        if wtype == TYPE_Q4_1:
            m = fp16_bits_to_f64(blk[..., 2:4].copy().view(np.uint16)[..., 0])
            v = d[..., None] * nibble_split_codes(blk[..., 4:20]) + m[..., None]
        elif wtype == TYPE_Q5_0:
            q = nibble_split_codes(blk[..., 6:22]) | (q5_high_bits(blk[..., 2:6]) << 4)
            v = d[..., None] * (q - 16)
        else:
            m = fp16_bits_to_f64(blk[..., 2:4].copy().view(np.uint16)[..., 0])
            q = nibble_split_codes(blk[..., 8:24]) | (q5_high_bits(blk[..., 4:8]) << 4)
            v = d[..., None] * q + m[..., None]
        return v.reshape(r, k)
    if wtype == TYPE_Q5_K:
        sb = rows.reshape(r, k // 256, 176)
        d = fp16_bits_to_f64(sb[..., 0:2].copy().view(np.uint16)[..., 0])
        dmin = fp16_bits_to_f64(sb[..., 2:4].copy().view(np.uint16)[..., 0])
        sc, mn = q4k_scale_min(sb[..., 4:16])
        q = q5k_codes(sb).reshape(r, k // 256, 8, 32).astype(np.float64)
        v = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None]
        return v.reshape(r, k)
    if wtype == TYPE_MXFP4:
        blk = rows.reshape(r, k // 32, 17)
        v = e2m1_value(nibble_split_codes(blk[..., 1:17])) * e8m0_value(blk[..., 0])[..., None]
        return v.reshape(r, k)
    raise ValueError(wtype)


# ---------------------------------------------------------------- integer block dots

def block_dots(wtype: int, rows, k: int, act_qs) -> np.ndarray:
    """Integer dot products per weight block of quantized rows against q8_1
    activation codes ``act_qs`` (int8 [k//32, 32]).

    Q8_0:  one int per 32-block, sum(w_q * a_q).
    NVFP4: one int per 16-block, sum((2*E2M1(code)) * a_q); doubling makes
           every E2M1 magnitude an integer {0,1,2,3,4,6,8,12}.
    Q4_K:  one int per 32-sub-block, sum(q4 * a_q).
    Q6_K:  one int per 16-value scale group, sum((q6 - 32) * a_q).
    Q4_0:  one int per 32-block, sum((q4 - 8) * a_q).
    Q4_1, Q5_1, Q5_K: one int per 32 values, sum(q * a_q) (q unsigned; the
           min term goes through the activation block's code sum).
    Q5_0:  one int per 32-block, sum((q5 - 16) * a_q).
    MXFP4: one int per 32-block, sum((2*E2M1(code)) * a_q).
    Returns int64 [R, nblocks]."""
    rows = np.asarray(rows, dtype=np.uint8)
    a = np.asarray(act_qs, dtype=np.int64).reshape(k)
    r = rows.shape[0]
    if wtype == TYPE_Q8_0:
        q = rows.reshape(r, k // 32, 34)[..., 2:34].view(np.int8).astype(np.int64)
        return (q * a.reshape(k // 32, 32)).sum(axis=-1)
    if wtype == TYPE_NVFP4:
        codes = rows[:, : k // 2].astype(np.int64)
        nib = np.stack([codes & 0x0F, codes >> 4], axis=-1).reshape(r, k)
        w2 = np.rint(2.0 * e2m1_value(nib)).astype(np.int64)
        return (w2 * a).reshape(r, k // 16, 16).sum(axis=-1)
    if wtype == TYPE_Q4_K:
        q = q4k_codes(rows.reshape(r, k // 256, 144)[..., 16:144]).reshape(r, k)
        return (q * a).reshape(r, k // 32, 32).sum(axis=-1)
    if wtype == TYPE_Q6_K:
        q = q6k_codes(rows.reshape(r, k // 256, 210)).reshape(r, k)
        return (q * a).reshape(r, k // 16, 16).sum(axis=-1)
    if wtype == TYPE_Q4_0:
        q = q4_0_codes(rows.reshape(r, k // 32, 18)).reshape(r, k)
        return (q * a).reshape(r, k // 32, 32).sum(axis=-1)
    if wtype == TYPE_Q4_1:
        q = nibble_split_codes(rows.reshape(r, k // 32, 20)[..., 4:20]).reshape(r, k)
    elif wtype == TYPE_Q5_0:
        blk = rows.reshape(r, k // 32, 22)
        q = (nibble_split_codes(blk[..., 6:22]) | (q5_high_bits(blk[..., 2:6]) << 4)).reshape(r, k) - 16
    elif wtype == TYPE_Q5_1:
        blk = rows.reshape(r, k // 32, 24)
        q = (nibble_split_codes(blk[..., 8:24]) | (q5_high_bits(blk[..., 4:8]) << 4)).reshape(r, k)
    elif wtype == TYPE_Q5_K:
        q = q5k_codes(rows.reshape(r, k // 256, 176)).reshape(r, k)
    elif wtype == TYPE_MXFP4:
        codes = nibble_split_codes(rows.reshape(r, k // 32, 17)[..., 1:17]).reshape(r, k)
        q = np.rint(2.0 * e2m1_value(codes)).astype(np.int64)
    else:
        raise ValueError(wtype)
    return (q * a).reshape(r, k // 32, 32).sum(axis=-1)
