"""Pins of the oracle's format codecs against things other than the oracle:
torch's float8 / bfloat16 decoders, exact rational arithmetic, hand-worked
golden blocks and brute force over Python ints."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F


# ---------------------------------------------------------------- float codecs

def test_ue4m3_matches_torch_e4m3fn_for_every_finite_code():
    codes = np.arange(0x7F, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(F.ue4m3_value(codes), ref)
    assert np.isnan(F.ue4m3_value(0x7F))
    assert np.isnan(F.ue4m3_value(0x80))          # sign bit is not part of UE4M3
    assert F.ue4m3_value(0x7E) == 448.0


def _e2m1_as_e4m3_bits(code: int) -> int:
    """E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit) embedded
    in E4M3 (bias 7): a normal E2M1 exponent e maps to field e + 6 and the
    mantissa bit to the top mantissa bit; subnormal 0.5 is 2^-1 (field 6)."""
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    if e == 0:
        bits = 0 if m == 0 else (6 << 3)
    else:
        bits = ((e + 6) << 3) | (m << 2)
    return (s << 7) | bits


def test_e2m1_matches_torch_through_e4m3_embedding():
    bits = np.array([_e2m1_as_e4m3_bits(c) for c in range(16)], dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e2m1_value(np.arange(16))
    assert np.array_equal(got, ref)
    assert list(np.abs(got[:8])) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_bf16_decode_matches_torch_all_codes():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = F.bf16_bits_to_f64(bits)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])


def test_round_to_bf16_matches_torch_on_fp32_inputs():
    r = np.random.default_rng(0)
    x = (r.standard_normal(200000) * np.exp2(r.integers(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.round_to_bf16(x.astype(np.float64)), ref)
    # exact midpoints between bf16 neighbours go to the even mantissa
    assert F.round_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert F.round_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


def test_ue4m3_encoder_matches_torch_rounding_including_ties():
    fin = F.ue4m3_value(np.arange(0x7F))
    mids = (fin[:-1] + fin[1:]) / 2.0                        # exact ties
    r = np.random.default_rng(1)
    vals = np.concatenate([mids, r.uniform(0, 448, 5000), r.uniform(0, 0.02, 5000), fin])
    vals = vals.astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.ue4m3_encode_rne_sat(vals), ref)
    assert F.ue4m3_encode_rne_sat(np.float32(1000.0)) == 0x7E


def test_e2m1_encoder_hand_table_and_brute_force():
    # hand-derived: ties go to the even code
    cases = {0.25: 0, 0.26: 1, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             5.01: 7, 7.0: 7, 100.0: 7, -0.1: 8, -5.0: 14, -6.0: 15, 0.0: 0}
    for v, c in cases.items():
        assert F.e2m1_encode_rne_sat(np.float32(v)) == c, v
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    r = np.random.default_rng(2)
    for v in r.uniform(-8, 8, 3000).astype(np.float32):
        a = abs(float(v))
        best = min(range(8), key=lambda i: (abs(table[i] - a), i % 2))
        assert F.e2m1_encode_rne_sat(v) == best | (8 if v < 0 else 0)


# ---------------------------------------------------------------- Q4_K

def test_q4k_scale_unpack_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q4k_scales.json")))
    sc, mn = F.q4k_scale_min(np.array(g["scales12"], dtype=np.uint8))
    assert list(sc) == g["sc"] and list(mn) == g["m"]


def test_q4k_scale_unpack_single_bit_bijection():
    """Each of the 96 bits lands in exactly one 6-bit field as a single bit,
    and all 16*6 (field, bit) slots are hit once."""
    hits = set()
    for byte in range(12):
        for bit in range(8):
            s = np.zeros(12, dtype=np.uint8)
            s[byte] = 1 << bit
            sc, mn = F.q4k_scale_min(s)
            fields = list(sc) + list(mn)
            nz = [(i, v) for i, v in enumerate(fields) if v]
            assert len(nz) == 1 and (nz[0][1] & (nz[0][1] - 1)) == 0
            hits.add((nz[0][0], int(nz[0][1]).bit_length() - 1))
    assert len(hits) == 96


def test_q4k_superblock_golden_values(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q4k_scales.json")))["superblock"]
    sb = np.zeros(144, dtype=np.uint8)
    sb[0:2] = np.array([g["d_bits"]], dtype=np.uint16).view(np.uint8)
    sb[2:4] = np.array([g["dmin_bits"]], dtype=np.uint16).view(np.uint8)
    sb[4:16] = json.load(open(os.path.join(golden_dir, "q4k_scales.json")))["scales12"]
    for c in range(4):
        for l in range(32):
            sb[16 + 32 * c + l] = (l % 16) | (((l + c) % 16) << 4)
    v = F.dequantize_rows(F.TYPE_Q4_K, sb[None, :], 256)[0]
    for idx, val in g["values"].items():
        assert v[int(idx)] == val, idx


def test_q6k_codes_single_bit_bijection():
    """With every code byte zero each code is -32; setting one bit of ql or qh
    raises exactly one code by a single power of two, and the 192*8 bits cover
    all 256*6 (value, bit) slots once."""
    hits = set()
    for byte in range(192):
        for bit in range(8):
            sb = np.zeros(210, dtype=np.uint8)
            sb[byte] = 1 << bit
            q = F.q6k_codes(sb) + 32
            nz = np.nonzero(q)[0]
            assert len(nz) == 1
            v = int(q[nz[0]])
            assert v & (v - 1) == 0
            hits.add((int(nz[0]), v.bit_length() - 1))
    assert len(hits) == 256 * 6


def test_q6k_superblock_hand_values():
    """Values worked by hand from the GGUF Q6_K layout (ql low 4 bits, qh high
    2 bits, int8 scale per 16 values, fp16 d; value d*scale*(q-32))."""
    sb = np.zeros(210, dtype=np.uint8)
    sb[208:210] = np.array([0x3800], dtype=np.uint16).view(np.uint8)   # d = 0.5
    sc = np.zeros(16, dtype=np.int8)
    sc[0], sc[2], sc[4], sc[6], sc[14] = 2, -1, 7, 1, -4
    sb[192:208] = sc.view(np.uint8)
    sb[0] = 0x21          # ql[0]: value 0 low bits 1, value 64 low bits 2
    sb[128] = 0x27        # qh[0]: value 0 high 3, value 32 high 1, value 64 high 2, value 96 high 0
    sb[64 + 32 + 5] = 0xF0  # ql[101]: value 229 low bits 15 (high nibble), value 165 low bits 0
    sb[128 + 32 + 5] = 0xC0  # qh[37]: value 229 high bits 3
    v = F.dequantize_rows(F.TYPE_Q6_K, sb[None, :], 256)[0]
    want = {0: 0.5 * 2 * (49 - 32), 32: 0.5 * -1 * (16 - 32), 64: 0.5 * 7 * (34 - 32), 96: 0.5 * 1 * -32,
            1: 0.5 * 2 * -32, 128: 0.0, 229: 0.5 * -4 * (63 - 32), 165: 0.0}
    for idx, val in want.items():
        assert v[idx] == val, (idx, v[idx], val)
    assert (17.0, 8.0, 7.0, -16.0, -32.0, -62.0) == (v[0], v[32], v[64], v[96], v[1], v[229])


def test_q4_0_codes_single_bit_and_hand_values():
    hits = set()
    for byte in range(2, 18):
        for bit in range(8):
            blk = np.zeros(18, dtype=np.uint8)
            blk[byte] = 1 << bit
            q = F.q4_0_codes(blk) + 8
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and (int(q[nz[0]]) & (int(q[nz[0]]) - 1)) == 0
            hits.add((int(nz[0]), int(q[nz[0]]).bit_length() - 1))
    assert len(hits) == 32 * 4
    blk = np.zeros(18, dtype=np.uint8)
    blk[0:2] = np.array([0x3400], dtype=np.uint16).view(np.uint8)   # d = 0.25
    blk[2] = 0x9F         # value 0: 15 - 8 = 7, value 16: 9 - 8 = 1
    v = F.dequantize_rows(F.TYPE_Q4_0, blk[None, :], 32)[0]
    assert (v[0], v[16], v[3], v[19]) == (1.75, 0.25, -2.0, -2.0)


def _f16(v):
    return np.array([v], dtype=np.float16).view(np.uint8)


@pytest.mark.parametrize("wtype,code_bytes,offset", [(F.TYPE_Q4_1, range(4, 20), 0),
                                                     (F.TYPE_Q5_0, range(2, 22), 16),
                                                     (F.TYPE_Q5_1, range(4, 24), 0)])
def test_q4_1_q5_codes_single_bit_bijection(wtype, code_bytes, offset):
    """d = 1, m = 0: each single set bit of the code and high-bit bytes gives
    exactly one value a single power-of-two code, and the bits cover every
    (value, code bit) pair once: 32 x 4 for Q4_1, 32 x 5 for Q5_x."""
    nb = F.row_bytes(wtype, 32)
    hits = set()
    for byte in code_bytes:
        for bit in range(8):
            blk = np.zeros(nb, dtype=np.uint8)
            blk[0:2] = _f16(1.0)
            blk[byte] = 1 << bit
            q = np.rint(F.dequantize_rows(wtype, blk[None, :], 32)[0]).astype(np.int64) + offset
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and (int(q[nz[0]]) & (int(q[nz[0]]) - 1)) == 0
            hits.add((int(nz[0]), int(q[nz[0]]).bit_length() - 1))
    assert len(hits) == 32 * (4 if wtype == F.TYPE_Q4_1 else 5)


def test_q4_1_q5_0_q5_1_hand_values():
    blk = np.zeros(20, dtype=np.uint8)                       # Q4_1: d = 0.5, m = -1
    blk[0:2], blk[2:4] = _f16(0.5), _f16(-1.0)
    blk[4] = 0x3A                                            # value 0: code 10, value 16: code 3
    v = F.dequantize_rows(F.TYPE_Q4_1, blk[None, :], 32)[0]
    assert (v[0], v[16], v[5]) == (4.0, 0.5, -1.0)
    blk = np.zeros(22, dtype=np.uint8)                       # Q5_0: d = 0.25, high bits of values 0 and 16
    blk[0:2] = _f16(0.25)
    blk[2:6] = np.array([0x00010001], dtype="<u4").view(np.uint8)
    blk[6] = 0x2F                                            # value 0: 15 + 16, value 16: 2 + 16
    v = F.dequantize_rows(F.TYPE_Q5_0, blk[None, :], 32)[0]
    assert (v[0], v[16], v[1]) == (3.75, 0.5, -4.0)
    blk = np.zeros(24, dtype=np.uint8)                       # Q5_1: d = 0.5, m = 0.25, high bit of value 31
    blk[0:2], blk[2:4] = _f16(0.5), _f16(0.25)
    blk[7] = 0x80
    blk[8 + 15] = 0x70                                       # value 15: code 0, value 31: 7 + 16
    v = F.dequantize_rows(F.TYPE_Q5_1, blk[None, :], 32)[0]
    assert (v[15], v[31]) == (0.25, 11.75)


def test_q5k_superblock_hand_values():
    """d = 1, dmin = 0.5; sub-block 0: sc 3, m 2; sub-block 5: sc 1 + 16
    (top bits from byte 1), m 2.  Value 0: nibble 5 + fifth bit (bit 0 of
    high-bit byte 0) = 21 -> 3*21 - 1 = 62.  Value 167 (sub-block 5, lane 7):
    high nibble 9 of code byte 64 + 7, fifth bit = bit 5 of high-bit byte 7
    -> 25 -> 17*25 - 1 = 424."""
    sb = np.zeros(176, dtype=np.uint8)
    sb[0:2], sb[2:4] = _f16(1.0), _f16(0.5)
    sb[4 + 0], sb[4 + 4] = 3, 2            # sc0, m0
    sb[4 + 1] = 0x40                       # top bits of sc5 = 1 (sc1 stays 0)
    sb[4 + 9] = 0x21                       # sc5 low nibble 1, m5 low nibble 2
    sb[48 + 0] = 0x05
    sb[16 + 0] = 0x01
    sb[48 + 64 + 7] = 0x90
    sb[16 + 7] = 0x20
    v = F.dequantize_rows(F.TYPE_Q5_K, sb[None, :], 256)[0]
    assert v[0] == 62.0 and v[167] == 424.0
    assert v[1] == -1.0                    # code 0 of sub-block 0: -dmin*m0
    assert v[160] == -1.0 and v[32] == 0.0  # sub-block 5 lane 0; sub-block 1 has sc = m = 0


def test_q5k_codes_single_bit_bijection():
    hits = set()
    for byte in range(16, 176):
        for bit in range(8):
            sb = np.zeros(176, dtype=np.uint8)
            sb[byte] = 1 << bit
            q = F.q5k_codes(sb)
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and (int(q[nz[0]]) & (int(q[nz[0]]) - 1)) == 0
            hits.add((int(nz[0]), int(q[nz[0]]).bit_length() - 1))
    assert len(hits) == 256 * 5


def test_mxfp4_codes_single_bit_bijection():
    """e = 127 (scale 1): each single set bit of the 16 code bytes changes
    exactly one value, to E2M1 of a one-bit code (0.5, 1, 2 or -0 for the
    sign bit alone), and the bits cover every (value, code bit) pair once."""
    hits = set()
    mags = {1: 0.5, 2: 1.0, 4: 2.0}
    for byte in range(1, 17):
        for bit in range(8):
            blk = np.zeros(17, dtype=np.uint8)
            blk[0] = 127
            blk[byte] = 1 << bit
            v = F.dequantize_rows(F.TYPE_MXFP4, blk[None, :], 32)[0]
            code_bit = bit % 4
            value = (byte - 1) + (16 if bit >= 4 else 0)
            if code_bit == 3:            # the sign bit of a zero code: -0
                assert (v == 0).all() and np.signbit(v[value]) and np.signbit(v).sum() == 1
            else:
                nz = np.nonzero(v)[0]
                assert list(nz) == [value] and v[value] == mags[1 << code_bit]
            hits.add((value, code_bit))
    assert len(hits) == 32 * 4


def test_mxfp4_hand_values_and_e8m0():
    assert F.e8m0_value(127) == 1.0 and F.e8m0_value(0) == 2.0 ** -127 and F.e8m0_value(254) == 2.0 ** 127
    blk = np.zeros(2 * 17, dtype=np.uint8)
    blk[0] = 126                            # 0.5
    blk[1] = 0x9B                           # value 0: code 11 = -1.5, value 16: code 9 = -0.5
    blk[17] = 130                           # 8
    blk[18 + 15] = 0x07                     # block 1 value 15: code 7 = 6
    v = F.dequantize_rows(F.TYPE_MXFP4, blk[None, :], 64)[0]
    assert (v[0], v[16], v[1]) == (-0.75, -0.25, 0.0)
    assert v[32 + 15] == 48.0 and v[32 + 31] == 0.0


# ---------------------------------------------------------------- q8_1

def _fp32_round(fr: Fraction) -> Fraction:
    """Round an exact rational to the nearest fp32 (ties to even), normal range."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (e - 23)                    # 24 significant bits
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def _round_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def test_q8_1_codes_match_exact_rational_reference():
    r = np.random.default_rng(3)
    x = (r.standard_normal((40, 32)) * np.exp2(r.integers(-8, 8, (40, 1)))).astype(np.float32)
    x[0, :] = 0
    x[1, :] = np.arange(32) - 16                                    # ramp
    qs, d_bits, s_bits, sumq = F.quantize_q8_1(x)
    for b in range(40):
        amax = max(abs(Fraction(float(v))) for v in x[b])
        d = _fp32_round(amax / 127)
        for i in range(32):
            want = 0 if d == 0 else _round_half_even(_fp32_round(Fraction(float(x[b, i])) / d))
            assert qs[b, 0, i] == want, (b, i)
        assert float(np.uint16(d_bits[b, 0]).view(np.float16)) == float(np.float16(float(d)))
        assert sumq[b, 0] == sum(int(v) for v in qs[b, 0])


def test_q8_1_golden_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q8_1_blocks.json")))
    qs, d, s, _ = F.quantize_q8_1(np.zeros(32, np.float32))
    assert not qs.any() and d[0] == 0 and s[0] == 0
    x = np.zeros(32, np.float32)
    x[5] = 3.0
    qs, d, s, _ = F.quantize_q8_1(x)
    spike = g["cases"][1]
    assert qs[0, 5] == spike["qs_at_5"] and np.count_nonzero(qs) == 1
    assert d[0] == spike["d_bits"] and s[0] == spike["s_bits"]


def test_q8_1_round_trip_bound():
    r = np.random.default_rng(4)
    x = r.standard_normal((500, 64)).astype(np.float32)
    qs, d_bits, _, _ = F.quantize_q8_1(x)
    back = F.dequantize_q8_1(qs, d_bits)
    xb = x.astype(np.float64).reshape(500, 2, 32)
    d32 = np.abs(xb).max(axis=-1) / 127.0
    dh = F.fp16_bits_to_f64(d_bits)
    bound = d32 / 2 * (1 + 1e-6) + 127 * np.abs(d32 - dh)
    err = np.abs(back.reshape(500, 2, 32) - xb).max(axis=-1)
    assert (err <= bound + 1e-12).all()


# ---------------------------------------------------------------- block dots

_E2M1_X2 = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 6, 6: 8, 7: 12}


@pytest.mark.parametrize("wtype,k", [(F.TYPE_Q8_0, 96), (F.TYPE_NVFP4, 128), (F.TYPE_Q4_K, 512),
                                     (F.TYPE_Q6_K, 512), (F.TYPE_Q4_0, 96), (F.TYPE_Q4_1, 96),
                                     (F.TYPE_Q5_0, 96), (F.TYPE_Q5_1, 96), (F.TYPE_Q5_K, 512),
                                     (F.TYPE_MXFP4, 96)])
def test_block_dots_brute_force(wtype, k):
    r = np.random.default_rng(5 + wtype)
    rb = F.row_bytes(wtype, k)
    rows = r.integers(0, 256, (3, rb), dtype=np.uint8)
    a = r.integers(-127, 128, (k // 32, 32)).astype(np.int8)
    got = F.block_dots(wtype, rows, k, a)
    af = [int(v) for v in a.reshape(-1)]
    for ri in range(3):
        row = [int(b) for b in rows[ri]]
        if wtype == F.TYPE_Q8_0:
            want = []
            for b in range(k // 32):
                blk = row[b * 34 + 2: b * 34 + 34]
                want.append(sum((v - 256 if v > 127 else v) * af[b * 32 + i] for i, v in enumerate(blk)))
        elif wtype == F.TYPE_NVFP4:
            vals = []
            for byte in row[: k // 2]:
                for nib in (byte & 15, byte >> 4):
                    mag = _E2M1_X2[nib & 7]
                    vals.append(-mag if nib & 8 else mag)
            want = [sum(vals[b * 16 + i] * af[b * 16 + i] for i in range(16)) for b in range(k // 16)]
        elif wtype == F.TYPE_Q6_K:
            vals = []
            for sbi in range(k // 256):
                b = row[sbi * 210: sbi * 210 + 210]
                for v in range(256):
                    n, c, l = v // 128, (v % 128) // 32, v % 32
                    lo = (b[64 * n + 32 * (c % 2) + l] >> (4 * (c // 2))) & 15
                    hi = (b[128 + 32 * n + l] >> (2 * c)) & 3
                    vals.append(lo + 16 * hi - 32)
            want = [sum(vals[g * 16 + i] * af[g * 16 + i] for i in range(16)) for g in range(k // 16)]
        elif wtype == F.TYPE_Q4_0:
            want = []
            for b in range(k // 32):
                qs = row[b * 18 + 2: b * 18 + 18]
                vals = [(x & 15) - 8 for x in qs] + [(x >> 4) - 8 for x in qs]
                want.append(sum(vals[i] * af[b * 32 + i] for i in range(32)))
        elif wtype in (F.TYPE_Q4_1, F.TYPE_Q5_0, F.TYPE_Q5_1, F.TYPE_MXFP4):
            nbytes, qoff, hoff = {F.TYPE_Q4_1: (20, 4, None), F.TYPE_Q5_0: (22, 6, 2), F.TYPE_Q5_1: (24, 8, 4),
                                  F.TYPE_MXFP4: (17, 1, None)}[wtype]
            want = []
            for b in range(k // 32):
                blk = row[b * nbytes: (b + 1) * nbytes]
                qs = blk[qoff: qoff + 16]
                vals = [x & 15 for x in qs] + [x >> 4 for x in qs]
                if hoff is not None:
                    word = blk[hoff] | (blk[hoff + 1] << 8) | (blk[hoff + 2] << 16) | (blk[hoff + 3] << 24)
                    vals = [v + 16 * ((word >> i) & 1) for i, v in enumerate(vals)]
                if wtype == F.TYPE_Q5_0:
                    vals = [v - 16 for v in vals]
                if wtype == F.TYPE_MXFP4:
                    vals = [(-_E2M1_X2[v & 7] if v & 8 else _E2M1_X2[v & 7]) for v in vals]
                want.append(sum(vals[i] * af[b * 32 + i] for i in range(32)))
        elif wtype == F.TYPE_Q5_K:
            want = []
            for sbi in range(k // 256):
                b = row[sbi * 176: sbi * 176 + 176]
                for j in range(8):
                    c = j // 2
                    codes = [((b[48 + c * 32 + l] >> (4 * (j % 2))) & 15) + 16 * ((b[16 + l] >> j) & 1)
                             for l in range(32)]
                    want.append(sum(codes[l] * af[sbi * 256 + j * 32 + l] for l in range(32)))
        else:
            want = []
            for sbi in range(k // 256):
                qs = row[sbi * 144 + 16: sbi * 144 + 144]
                for j in range(8):
                    c = j // 2
                    codes = [(qs[c * 32 + l] >> (4 * (j % 2))) & 15 for l in range(32)]
                    base = sbi * 256 + j * 32
                    want.append(sum(codes[l] * af[base + l] for l in range(32)))
        assert list(got[ri]) == want


def test_f16_f32_rows_hand_values():
    """Little-endian fp16 / fp32 rows decode to their IEEE values: 1, -2,
    the smallest fp16 subnormal 2^-24, the largest fp16 65504; fp32 1.5,
    -0.25, 2^-149."""
    h = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF] * 8, dtype="<u2").view(np.uint8)
    v = F.dequantize_rows(F.TYPE_F16, h[None, :], 32)[0]
    assert list(v[:4]) == [1.0, -2.0, 2.0 ** -24, 65504.0]
    f = np.array([0x3FC00000, 0xBE800000, 0x00000001, 0] * 8, dtype="<u4").view(np.uint8)
    v = F.dequantize_rows(F.TYPE_F32, f[None, :], 32)[0]
    assert list(v[:4]) == [1.5, -0.25, 2.0 ** -149, 0.0]
    assert F.row_bytes(F.TYPE_F16, 64) == 128 and F.row_bytes(F.TYPE_F32, 64) == 256


def test_row_bytes_match_the_pages_geometry():
    # FreeToken issue #194, Reproduction geometry: Q4_K 3,538,944 B gate/up and
    # 1,769,472 B down per expert; BF16 12,582,912 B and 6,291,456 B (H=4096, I=768)
    H, I = 4096, 768
    assert 2 * I * F.row_bytes(F.TYPE_Q4_K, H) == 3538944
    assert H * F.row_bytes(F.TYPE_Q4_K, I) == 1769472
    assert 2 * I * F.row_bytes(F.TYPE_BF16, H) == 12582912
    assert H * F.row_bytes(F.TYPE_BF16, I) == 6291456
    assert F.row_bytes(F.TYPE_NVFP4, 2048) == 1152 and F.row_bytes(F.TYPE_Q8_0, 256) == 272
    assert F.row_bytes(F.TYPE_Q4_K, 100) == 0
