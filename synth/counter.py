"""Counter-based bank bytes from SplitMix64, on the host (numpy) and on the GPU (torch).

SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): the n-th output (n >= 0) of the stream with seed s
is mix(s + (n + 1) * 0x9E3779B97F4A7C15 mod 2^64) where
mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
z *= 0x94D049BB133111EB; z ^= z >> 31  (all mod 2^64, logical shifts).

Byte o of a bank with seed s is byte (o mod 8) (little-endian) of output
o // 8.  Then a per-format mask, a function of the byte's position inside its
row only, keeps scale fields finite and of a realistic size:

  NVFP4 (row = K/2 code bytes, K/16 UE4M3 bytes): scale byte b -> 0x30 | (b & 0x0F)
        (exponent field 6 or 7: scales 0.5 .. 1.875); code bytes unchanged.
  Q4_K (144-byte super-blocks): d fp16 -> exponent field 1 (2^-14 .. 2^-13),
        dmin fp16 -> exponent field 4 (2^-11 .. 2^-10); the rest unchanged.
  Q8_0 (34-byte blocks): d fp16 -> exponent field 3 (2^-12 .. 2^-11);
        code byte 0x80 (-128) -> 0x81 (-127).
  Q6_K (210-byte super-blocks): the 16 int8 sub-block scales keep their low 5
        bits (0 .. 31); d fp16 -> exponent field 1 (2^-14 .. 2^-13).
  Q4_0 (18-byte blocks): d fp16 -> exponent field 3 (2^-12 .. 2^-11).
  Q4_1 / Q5_1 (20 / 24-byte blocks): d as Q4_0; m fp16 keeps its sign,
        exponent field 3.  Q5_0 (22-byte blocks): d as Q4_0.
  Q5_K (176-byte super-blocks): d and dmin as Q4_K.
  MXFP4 (17-byte blocks): E8M0 byte -> 118 + (b & 3) (scales 2^-9 .. 2^-6).
  BF16: each value keeps its sign and 7 mantissa bits; its exponent becomes
        119 + (bits 7..8 of the raw value): magnitudes 2^-8 .. 2^-4.
  F16: each value keeps its sign and 10 mantissa bits; its exponent field
        becomes 7 + (bits 10..11): magnitudes 2^-8 .. 2^-4.
  F32: each value keeps its sign and 23 mantissa bits; its exponent field
        becomes 119 + (bits 23..24): magnitudes 2^-8 .. 2^-4.

Both implementations below follow this definition independently.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB
M64 = (1 << 64) - 1

BF16, Q8_0, Q4_K, NVFP4, Q6_K, Q4_0 = 0, 1, 2, 3, 4, 5
Q4_1, Q5_0, Q5_1, Q5_K, MXFP4 = 6, 7, 8, 9, 10
F16, F32 = 11, 12


def _row_bytes(wtype: int, k: int) -> int:
    return {BF16: 2 * k, Q8_0: k // 32 * 34, Q4_K: k // 256 * 144, NVFP4: k // 2 + k // 16,
            Q6_K: k // 256 * 210, Q4_0: k // 32 * 18, Q4_1: k // 32 * 20, Q5_0: k // 32 * 22,
            Q5_1: k // 32 * 24, Q5_K: k // 256 * 176, MXFP4: k // 32 * 17, F16: 2 * k, F32: 4 * k}[wtype]


# ------------------------------------------------------------------ host (numpy)

def words_np(seed: int, first: int, count: int) -> np.ndarray:
    n = np.arange(first, first + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & M64) + (n + np.uint64(1)) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(C2)
        z = z ^ (z >> np.uint64(31))
    return z


def bank_bytes_np(seed: int, wtype: int, k: int, row0: int, nrows: int) -> np.ndarray:
    """Rows [row0, row0 + nrows) of the counter-based bank (rows of ``k``
    values of ``wtype``), as uint8 [nrows, row_bytes]."""
    rb = _row_bytes(wtype, k)
    b0, b1 = row0 * rb, (row0 + nrows) * rb
    w0, w1 = b0 // 8, (b1 + 7) // 8
    raw = words_np(seed, w0, w1 - w0).view(np.uint8)
    out = raw[b0 - w0 * 8: b0 - w0 * 8 + (b1 - b0)].reshape(nrows, rb).copy()
    return _mask_np(out, wtype, k)


def _mask_np(rows: np.ndarray, wtype: int, k: int) -> np.ndarray:
    if wtype == NVFP4:
        s = rows[:, k // 2:]
        rows[:, k // 2:] = 0x30 | (s & 0x0F)
    elif wtype == Q4_K:
        sb = rows.reshape(rows.shape[0], -1, 144)
        sb[..., 1] = 0x04 | (sb[..., 1] & 0x03)
        sb[..., 3] = 0x10 | (sb[..., 3] & 0x03)
    elif wtype == Q8_0:
        blk = rows.reshape(rows.shape[0], -1, 34)
        blk[..., 1] = 0x0C | (blk[..., 1] & 0x03)
        q = blk[..., 2:]
        q[q == 0x80] = 0x81
    elif wtype == Q6_K:
        sb = rows.reshape(rows.shape[0], -1, 210)
        sb[..., 192:208] &= 0x1F
        sb[..., 209] = 0x04 | (sb[..., 209] & 0x03)
    elif wtype == Q4_0:
        blk = rows.reshape(rows.shape[0], -1, 18)
        blk[..., 1] = 0x0C | (blk[..., 1] & 0x03)
    elif wtype in (Q4_1, Q5_0, Q5_1):
        blk = rows.reshape(rows.shape[0], -1, {Q4_1: 20, Q5_0: 22, Q5_1: 24}[wtype])
        blk[..., 1] = 0x0C | (blk[..., 1] & 0x03)
        if wtype != Q5_0:
            blk[..., 3] = (blk[..., 3] & 0x80) | 0x0C | (blk[..., 3] & 0x03)
    elif wtype == Q5_K:
        sb = rows.reshape(rows.shape[0], -1, 176)
        sb[..., 1] = 0x04 | (sb[..., 1] & 0x03)
        sb[..., 3] = 0x10 | (sb[..., 3] & 0x03)
    elif wtype == MXFP4:
        blk = rows.reshape(rows.shape[0], -1, 17)
        blk[..., 0] = 118 + (blk[..., 0] & 0x03)
    elif wtype == BF16:
        v = rows.view(np.uint16).astype(np.uint32)
        exp = 119 + ((v >> 7) & 3)
        v = (v & 0x807F) | (exp << 7)
        rows[:] = v.astype(np.uint16).view(np.uint8).reshape(rows.shape)
    elif wtype == F16:
        v = rows.view(np.uint16).astype(np.uint32)
        exp = 7 + ((v >> 10) & 3)
        v = (v & 0x83FF) | (exp << 10)
        rows[:] = v.astype(np.uint16).view(np.uint8).reshape(rows.shape)
    elif wtype == F32:
        v = rows.view(np.uint32).astype(np.uint64)
        exp = 119 + ((v >> 23) & 3)
        v = (v & 0x807FFFFF) | (exp << 23)
        rows[:] = v.astype(np.uint32).view(np.uint8).reshape(rows.shape)
    return rows


# ------------------------------------------------------------------ device (torch)

def _s64(c: int) -> int:
    """The int64 with the same 64 bits as the unsigned constant ``c``."""
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(z, s: int):
    import torch
    return torch.bitwise_and(torch.bitwise_right_shift(z, s), (1 << (64 - s)) - 1)


def fill_bank_torch(dst, seed: int, wtype: int, k: int, chunk_rows: int | None = None) -> None:
    """Fill the uint8 CUDA (or CPU) tensor ``dst`` (a whole number of rows of
    ``k`` values of ``wtype``; its size a multiple of 8 bytes) with the
    counter-based bank of ``seed``.  Works chunk by chunk to bound the
    temporaries."""
    import torch
    rb = _row_bytes(wtype, k)
    total = dst.numel()
    assert total % rb == 0 and total % 8 == 0
    nrows = total // rb
    if chunk_rows is None:
        chunk_rows = max(8, (1 << 28) // rb // 8 * 8)    # ~256 MiB of rows, even count
    chunk_rows = max(8, chunk_rows // 8 * 8)                # keeps chunk starts 8-byte aligned
    words = dst.view(torch.int64)
    g = _s64(GAMMA)
    c1, c2 = _s64(C1), _s64(C2)
    for r0 in range(0, nrows, chunk_rows):
        r1 = min(nrows, r0 + chunk_rows)
        wb0, wb1 = r0 * rb // 8, (r1 * rb + 7) // 8
        n = torch.arange(wb0, wb1, dtype=torch.int64, device=dst.device)
        z = (n + 1) * g + _s64(seed & M64)
        z = torch.bitwise_xor(z, _lsr(z, 30)) * c1
        z = torch.bitwise_xor(z, _lsr(z, 27)) * c2
        z = torch.bitwise_xor(z, _lsr(z, 31))
        words[wb0:wb1] = z
        del n, z
        rows = dst[r0 * rb: r1 * rb].view(r1 - r0, rb)
        _mask_torch(rows, wtype, k)


def _mask_torch(rows, wtype: int, k: int) -> None:
    import torch
    if wtype == NVFP4:
        s = rows[:, k // 2:]
        s.copy_(torch.bitwise_or(torch.bitwise_and(s, 0x0F), 0x30))
    elif wtype == Q4_K:
        sb = rows.view(rows.shape[0], -1, 144)
        sb[..., 1] = torch.bitwise_or(torch.bitwise_and(sb[..., 1], 0x03), 0x04)
        sb[..., 3] = torch.bitwise_or(torch.bitwise_and(sb[..., 3], 0x03), 0x10)
    elif wtype == Q8_0:
        blk = rows.view(rows.shape[0], -1, 34)
        blk[..., 1] = torch.bitwise_or(torch.bitwise_and(blk[..., 1], 0x03), 0x0C)
        q = blk[..., 2:]
        q.masked_fill_(q == 0x80, 0x81)
    elif wtype == Q6_K:
        sb = rows.view(rows.shape[0], -1, 210)
        sb[..., 192:208] = torch.bitwise_and(sb[..., 192:208], 0x1F)
        sb[..., 209] = torch.bitwise_or(torch.bitwise_and(sb[..., 209], 0x03), 0x04)
    elif wtype == Q4_0:
        blk = rows.view(rows.shape[0], -1, 18)
        blk[..., 1] = torch.bitwise_or(torch.bitwise_and(blk[..., 1], 0x03), 0x0C)
    elif wtype in (Q4_1, Q5_0, Q5_1):
        blk = rows.view(rows.shape[0], -1, {Q4_1: 20, Q5_0: 22, Q5_1: 24}[wtype])
        blk[..., 1] = torch.bitwise_or(torch.bitwise_and(blk[..., 1], 0x03), 0x0C)
        if wtype != Q5_0:
            blk[..., 3] = torch.bitwise_or(torch.bitwise_and(blk[..., 3], 0x83), 0x0C)
    elif wtype == Q5_K:
        sb = rows.view(rows.shape[0], -1, 176)
        sb[..., 1] = torch.bitwise_or(torch.bitwise_and(sb[..., 1], 0x03), 0x04)
        sb[..., 3] = torch.bitwise_or(torch.bitwise_and(sb[..., 3], 0x03), 0x10)
    elif wtype == MXFP4:
        blk = rows.view(rows.shape[0], -1, 17)
        blk[..., 0] = torch.bitwise_and(blk[..., 0], 0x03) + 118
    elif wtype == BF16:
        v = rows.view(torch.int16).to(torch.int32) & 0xFFFF
        exp = 119 + torch.bitwise_and(torch.bitwise_right_shift(v, 7), 3)
        v = torch.bitwise_or(torch.bitwise_and(v, 0x807F), torch.bitwise_left_shift(exp, 7))
        v = torch.where(v >= 0x8000, v - 0x10000, v)
        rows.view(torch.int16).copy_(v.to(torch.int16))
    elif wtype == F16:
        v = rows.view(torch.int16).to(torch.int32) & 0xFFFF
        exp = 7 + torch.bitwise_and(torch.bitwise_right_shift(v, 10), 3)
        v = torch.bitwise_or(torch.bitwise_and(v, 0x83FF), torch.bitwise_left_shift(exp, 10))
        v = torch.where(v >= 0x8000, v - 0x10000, v)
        rows.view(torch.int16).copy_(v.to(torch.int16))
    elif wtype == F32:
        v = rows.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
        exp = 119 + torch.bitwise_and(torch.bitwise_right_shift(v, 23), 3)
        v = torch.bitwise_or(torch.bitwise_and(v, 0x807FFFFF), torch.bitwise_left_shift(exp, 23))
        v = torch.where(v >= 0x80000000, v - 0x100000000, v)
        rows.view(torch.int32).copy_(v.to(torch.int32))
