// Block formats of the expert banks and activations, as device functions.
//
// One "block" is 32 consecutive values of a row (8 for BF16 rows).  Each
// quantized type decodes a block into int8x4 words that line up with the
// q8_1 activation words, so the integer part of a block dot is a run of
// dp4a instructions; the float part applies the block scales.  These are the
// only definitions of the formats on the GPU side: the decode kernels and the
// block-dot test hook both call them.
//
// Formats (FreeToken PR #704, "How it plugs into the CPU executor";
// FreeToken issue #194, "Reproduction geometry"; Strata PR #292,
// "Summary/Pipeline"):
//   q8_1  : 32 int8 q, fp16 d, fp16 s; value q*d.
//   Q8_0  : fp16 d then 32 int8 (34 bytes); value d*q.
//   Q4_K  : 144-byte super-block of 256: fp16 d, fp16 dmin, 12 packed 6-bit
//           (sc, m) bytes, 128 code bytes; value d*sc_j*q - dmin*m_j.
//   NVFP4 : row = K/2 E2M1 code bytes (element 2i low nibble of byte i) then
//           K/16 UE4M3 scale bytes; value E2M1(code)*UE4M3(scale).
//   Q6_K  : 210-byte super-block of 256: ql[128] (low 4 bits), qh[64] (high
//           2 bits), 16 int8 scales (one per 16 values), fp16 d;
//           value d*sc_g*(q - 32).
//   Q4_0  : fp16 d then 16 code bytes (18 bytes per 32 values); value j < 16
//           is the low nibble of code byte j, value j+16 its high nibble;
//           value d*(q - 8).
//   Q4_1  : fp16 d, fp16 m, 16 code bytes as Q4_0 (20 bytes); value d*q + m.
//   Q5_0  : fp16 d, a 32-bit word whose bit j is the fifth code bit of value
//           j, 16 code bytes as Q4_0 (22 bytes); value d*(q - 16).
//   Q5_1  : fp16 d, fp16 m, the high-bit word, 16 code bytes (24 bytes);
//           value d*q + m.
//   Q5_K  : 176-byte super-block of 256: the Q4_K header (d, dmin, 12 packed
//           scale bytes), 32 high-bit bytes (bit j of byte l: value l of
//           sub-block j), 128 code bytes as Q4_K; value d*sc_j*q - dmin*m_j.
//   MXFP4 : one E8M0 byte e, 16 code bytes of E2M1 as Q4_0 (17 bytes);
//           value E2M1(code) * 2^(e - 127).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace qre {

enum WType : int {
  W_BF16 = 0, W_Q8_0 = 1, W_Q4_K = 2, W_NVFP4 = 3, W_Q6_K = 4, W_Q4_0 = 5,
  W_Q4_1 = 6, W_Q5_0 = 7, W_Q5_1 = 8, W_Q5_K = 9, W_MXFP4 = 10, W_F16 = 11, W_F32 = 12
};
// Float rows (BF16, F16, F32): the activations reach them unquantized.
__host__ __device__ constexpr bool is_float_w(int t) { return t == W_BF16 || t == W_F16 || t == W_F32; }
// Kernel-side variant of W_NVFP4 whose rows (9k/16 bytes) are not 16-byte aligned.
constexpr int W_NVFP4_U = 16;

__host__ __device__ inline int row_bytes_of(int t, int k) {
  switch (t) {
    case W_BF16: return (k % 32 == 0) ? 2 * k : 0;
    case W_Q8_0: return (k % 32 == 0) ? (k / 32) * 34 : 0;
    case W_Q4_K: return (k % 256 == 0) ? (k / 256) * 144 : 0;
    case W_NVFP4: return (k % 32 == 0) ? k / 2 + k / 16 : 0;
    case W_Q6_K: return (k % 256 == 0) ? (k / 256) * 210 : 0;
    case W_Q4_0: return (k % 32 == 0) ? (k / 32) * 18 : 0;
    case W_Q4_1: return (k % 32 == 0) ? (k / 32) * 20 : 0;
    case W_Q5_0: return (k % 32 == 0) ? (k / 32) * 22 : 0;
    case W_Q5_1: return (k % 32 == 0) ? (k / 32) * 24 : 0;
    case W_Q5_K: return (k % 256 == 0) ? (k / 256) * 176 : 0;
    case W_MXFP4: return (k % 32 == 0) ? (k / 32) * 17 : 0;
    case W_F16: return (k % 32 == 0) ? 2 * k : 0;
    case W_F32: return (k % 32 == 0) ? 4 * k : 0;
  }
  return 0;
}

// ------------------------------------------------------------------ q8_1

// A q8_1 activation block as the dot loops hold it: the 32 codes as eight
// int8x4 words in value order, d decoded from its fp16 copy, and the exact
// integer sum of the codes (for the Q4_K min and the Q4_0 offset terms).
struct ActQ8 {
  int q[8];
  float d;
  int sum;
};

// The exact path of the q8_1 rule for one element: rint(x / d) with the IEEE
// division, 0 when d == 0.  It is taken rarely (x*r within 2^-12 of a
// half-integer, or d not a normal number), so it stays out of line: inlined
// at every element it would multiply the code size of each quantizing kernel.
static __device__ __noinline__ int q8_1_code_exact(float x, float d) {
  return (d == 0.0f) ? 0 : __float2int_rn(__fdiv_rn(x, d));
}

// Quantize one 32-value block held by one thread: d = amax/127 (IEEE fp32
// division), q_i = round-half-even(v_i/d) (IEEE fp32 division), 0 when d = 0;
// returns the 32 codes packed as eight int8x4 words, d, and the exact code
// sum.  Every q8_1 quantization on the GPU (activations, the intermediate and
// the test hook) goes through this function.
//
// The codes are computed as rint(v * r) with r = 1/d rounded to nearest.
// |v*r - v/d| <= 2^-23 * |v/d| + ulp <= 2^-16 here (|v/d| <= 127), so the
// rounding to an integer can only differ from rint(v/d) when v*r lies within
// 2^-12 of a half-integer; such elements (and blocks whose d is not a normal
// number) take the IEEE division itself.
__device__ __forceinline__ void q8_1_quantize_block(const float (&v)[32], uint32_t (&qw)[8], float& d, int& sum) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  d = __fdiv_rn(amax, 127.0f);
  const bool fast = d >= 1.1754944e-38f;   // normal d: r is finite and accurate
  const float r = fast ? __frcp_rn(d) : 0.0f;
  sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x = v[4 * w + j];
      const float t = x * r;
      const float near = fabsf(t - floorf(t) - 0.5f);
      int q;
      if (fast && near > 0.000244140625f) q = __float2int_rn(t);
      else q = q8_1_code_exact(x, d);
      sum += q;
      word |= ((uint32_t)(q & 0xFF)) << (8 * j);
    }
    qw[w] = word;
  }
}

// The same q8_1 rule with a block spread over a lane quad (lanes 4k..4k+3 of
// a full warp), each lane holding 8 consecutive values (v[i] is value
// 8*(lane&3)+i of the block): amax and the code sum are combined with
// shuffles; w0/w1 receive this lane's 8 codes as two int8x4 words.
__device__ __forceinline__ void q8_1_quantize_quad(const float (&v)[8], uint32_t& w0, uint32_t& w1, float& d,
                                                   int& sum) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  d = __fdiv_rn(amax, 127.0f);
  const bool fast = d >= 1.1754944e-38f;
  const float r = fast ? __frcp_rn(d) : 0.0f;
  int s = 0;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float t = v[i] * r;
    const float near = fabsf(t - floorf(t) - 0.5f);
    int q;
    if (fast && near > 0.000244140625f) q = __float2int_rn(t);
    else q = q8_1_code_exact(v[i], d);
    s += q;
    w[i >> 2] |= ((uint32_t)(q & 0xFF)) << (8 * (i & 3));
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  w0 = w[0];
  w1 = w[1];
  sum = s;
}

// The same q8_1 rule with a block spread over a full warp, one value per
// lane (lane i holds value i of the block): amax and the code sum are
// combined with shuffles; returns this lane's code.
__device__ __forceinline__ int q8_1_quantize_lane(float v, float& d, int& sum) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  d = __fdiv_rn(amax, 127.0f);
  const bool fast = d >= 1.1754944e-38f;
  const float r = fast ? __frcp_rn(d) : 0.0f;
  const float t = v * r;
  const float near = fabsf(t - floorf(t) - 0.5f);
  int q;
  if (fast && near > 0.000244140625f) q = __float2int_rn(t);
  else q = q8_1_code_exact(v, d);
  int s = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  sum = s;
  return q;
}

// Internal q8_1 storage is planar: codes [rows][n] int8, d [rows][n/32] fp32
// (an fp16 value), exact code sum [rows][n/32] int32, s [rows][n/32] fp16 bits.
__device__ __forceinline__ ActQ8 load_act_q8(const int8_t* q, const float* d, const int* sum, size_t row_vals,
                                             size_t row_blocks, int blk) {
  ActQ8 a;
  const int4* p = reinterpret_cast<const int4*>(q + row_vals + 32 * (size_t)blk);
  const int4 lo = __ldg(p), hi = __ldg(p + 1);
  a.q[0] = lo.x; a.q[1] = lo.y; a.q[2] = lo.z; a.q[3] = lo.w;
  a.q[4] = hi.x; a.q[5] = hi.y; a.q[6] = hi.z; a.q[7] = hi.w;
  a.d = __ldg(d + row_blocks + blk);
  a.sum = __ldg(sum + row_blocks + blk);
  return a;
}

// ------------------------------------------------------------------ NVFP4

// |2*E2M1| for codes 0..7 as bytes: {0,1,2,3,4,6,8,12}.
constexpr uint32_t kE2M1x2Lo = 0x03020100u;
constexpr uint32_t kE2M1x2Hi = 0x0C080604u;

// The 32 codes of one block (16 bytes, element 2i in the low nibble of byte
// i) as magnitude words split by sign: pos[w] holds |2*value| of the
// non-negative codes of elements 4w..4w+3 (0 for negative codes), neg[w]
// those of the negative codes.  The split comes free from prmt: a selector
// nibble with its top bit set yields the replicated sign of a non-negative
// table byte, i.e. 0.
__device__ __forceinline__ void nvfp4_words(const uint4 c, uint32_t (&pos)[8], uint32_t (&neg)[8]) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t qv = cw[w], qx = qv ^ 0x88888888u;
    pos[2 * w] = prmt(kE2M1x2Lo, kE2M1x2Hi, qv);
    neg[2 * w] = prmt(kE2M1x2Lo, kE2M1x2Hi, qx);
    pos[2 * w + 1] = prmt(kE2M1x2Lo, kE2M1x2Hi, qv >> 16);
    neg[2 * w + 1] = prmt(kE2M1x2Lo, kE2M1x2Hi, qx >> 16);
  }
}

// Decode the 32 codes of block b of a row (see nvfp4_words) and the UE4M3
// scales of its two 16-value halves.
// A row is 9k/16 bytes: 16-byte aligned when k is a multiple of 256, else
// only 2-byte aligned, and then (kAligned false) the codes are gathered 2
// bytes at a time.
template <bool kAligned = true>
__device__ __forceinline__ void nvfp4_decode(const uint8_t* row, int k, int b, uint32_t (&pos)[8],
                                             uint32_t (&neg)[8], float2& scales) {
  const uint8_t* cp = row + 16 * b;
  uint4 c;
  if constexpr (kAligned) {
    c = lds128(cp);
  } else {
    c.x = lds16(cp) | ((uint32_t)lds16(cp + 2) << 16);
    c.y = lds16(cp + 4) | ((uint32_t)lds16(cp + 6) << 16);
    c.z = lds16(cp + 8) | ((uint32_t)lds16(cp + 10) << 16);
    c.w = lds16(cp + 12) | ((uint32_t)lds16(cp + 14) << 16);
  }
  nvfp4_words(c, pos, neg);
  scales = ue4m3x2_to_float2(lds16(row + (k >> 1) + 2 * b));
}

// The same codes as signed bytes (2*value in -12..12): a negative code's
// magnitude n becomes (0x80 - n) ^ 0x80 = 256 - n, computed on whole words
// without borrows (n <= 12 < 0x80), and the positive and negative halves
// are disjoint.  One dp4a per word and token instead of two: the cheaper
// form once a decoded block is dotted with three or more tokens.
__device__ __forceinline__ void nvfp4_signed(const uint32_t (&pos)[8], const uint32_t (&neg)[8], int (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = (int)(pos[i] | ((0x80808080u - neg[i]) ^ 0x80808080u));
}

// Integer dots of the two 16-value halves: sum((2*E2M1) * q).
__device__ __forceinline__ void nvfp4_int_dots(const uint32_t (&pos)[8], const uint32_t (&neg)[8], const int (&q)[8],
                                               int& d0, int& d1) {
  int p0 = 0, n0 = 0, p1 = 0, n1 = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    p0 = __dp4a((int)pos[w], q[w], p0);
    n0 = __dp4a((int)neg[w], q[w], n0);
    p1 = __dp4a((int)pos[w + 4], q[w + 4], p1);
    n1 = __dp4a((int)neg[w + 4], q[w + 4], n1);
  }
  d0 = p0 - n0;
  d1 = p1 - n1;
}

// ------------------------------------------------------------------ Q4_K

// d*sc_j and dmin*m_j of sub-block j from the 16-byte header of a Q4_K or
// Q5_K super-block (x: d | dmin << 16, y: scales[0..3], z: scales[4..7],
// w: scales[8..11]); both products are exact in fp32.
__device__ __forceinline__ void k_quant_scales(const uint4 hdr, int j, float& dsc, float& dmm) {
  const float d = f16_bits_to_f32(hdr.x & 0xFFFFu);
  const float dmin = f16_bits_to_f32(hdr.x >> 16);
  uint32_t sc, m;
  if (j < 4) {
    sc = (hdr.y >> (8 * j)) & 63u;
    m = (hdr.z >> (8 * j)) & 63u;
  } else {
    const int jj = j - 4;
    const uint32_t s8 = (hdr.w >> (8 * jj)) & 0xFFu;
    sc = (s8 & 15u) | (((hdr.y >> (8 * jj + 6)) & 3u) << 4);
    m = (s8 >> 4) | (((hdr.z >> (8 * jj + 6)) & 3u) << 4);
  }
  dsc = d * (float)sc;
  dmm = dmin * (float)m;
}

// Decode sub-block b (32 values) of a Q4_K row: the codes as int8x4 words in
// value order, and the fp32 factors d*sc_j and dmin*m_j (both exact).
__device__ __forceinline__ void q4k_decode(const uint8_t* row, int b, int (&nib)[8], float& dsc, float& dmm) {
  const uint8_t* sb = row + (b >> 3) * 144;
  const int j = b & 7;
  k_quant_scales(lds128(sb), j, dsc, dmm);
  const uint8_t* qs = sb + 16 + (j >> 1) * 32;
  const uint4 q0 = lds128(qs), q1 = lds128(qs + 16);
  const int sh = (j & 1) * 4;
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) nib[i] = (int)((w[i] >> sh) & 0x0F0F0F0Fu);
}

// Sub-block b of a Q5_K row (16-byte aligned super-blocks): the 5-bit codes
// as int8x4 words in value order and d*sc_j, dmin*m_j.  The low 4 bits are
// laid out as in Q4_K (code bytes at offset 48); the fifth bit of value l is
// bit j of high-bit byte l (offset 16).
__device__ __forceinline__ void q5k_decode(const uint8_t* row, int b, int (&q)[8], float& dsc, float& dmm) {
  const uint8_t* sb = row + (b >> 3) * 176;
  const int j = b & 7;
  k_quant_scales(lds128(sb), j, dsc, dmm);
  const uint8_t* qs = sb + 48 + (j >> 1) * 32;
  const uint4 q0 = lds128(qs), q1 = lds128(qs + 16);
  const uint4 h0 = lds128(sb + 16), h1 = lds128(sb + 32);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const uint32_t h[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  const int sh = (j & 1) * 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = (int)(((w[i] >> sh) & 0x0F0F0F0Fu) | (((h[i] >> j) & 0x01010101u) << 4));
}

__device__ __forceinline__ int int_dot8(const int (&w)[8], const int (&q)[8]) {
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = __dp4a(w[i], q[i], s);
  return s;
}

// ------------------------------------------------------------------ Q8_0

// Block b of a Q8_0 row (34-byte blocks, 2-byte aligned in shared memory).
__device__ __forceinline__ void q8_0_decode(const uint8_t* row, int b, int (&w)[8], float& d) {
  const uint8_t* blk = row + 34 * b;
  d = f16_bits_to_f32(lds16(blk));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = lds16(blk + 2 + 4 * i), hi = lds16(blk + 4 + 4 * i);
    w[i] = (int)(lo | (hi << 16));
  }
}

// ------------------------------------------------------------------ Q6_K

// 32 bytes from a 2-byte aligned address inside a super-block as eight
// words: aligned 32-bit loads, realigned with a funnel shift when the address
// is 2 mod 4.  The extra word read then ends 2 bytes past the 32, which every
// caller keeps inside the same super-block.
__device__ __forceinline__ void lds_words8_a2(const uint8_t* p, uint32_t (&w)[8]) {
  const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);  // 0 or 2
  const uint8_t* a = p - mis;
  uint32_t r[9];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = lds32(a + 4 * i);
  r[8] = mis ? lds32(a + 32) : 0u;
  const uint32_t sh = 8u * mis;
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], sh);
}

// Decode sub-block b (32 values) of a Q6_K row (super-blocks 2-byte aligned):
// the signed codes q - 32 as int8x4 words in value order, d, and the two
// int8 scales of its 16-value halves.  Sub-block j = b mod 8 of a super-block
// covers values 32j .. 32j+31, i.e. half n = j/4 and quarter c = j mod 4: its
// low nibbles are nibble c/2 of ql[64n + 32(c mod 2) + l] and its high bits
// are bits 2c, 2c+1 of qh[32n + l], l = 0..31.
__device__ __forceinline__ void q6k_decode(const uint8_t* row, int b, int (&w)[8], float& d, float& s0, float& s1) {
  const uint8_t* sb = row + (b >> 3) * 210;
  const int j = b & 7, n = j >> 2, c = j & 3;
  uint32_t lo[8], hi[8];
  lds_words8_a2(sb + 64 * n + 32 * (c & 1), lo);
  lds_words8_a2(sb + 128 + 32 * n, hi);
  const int sl = 4 * (c >> 1), sh = 2 * c;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // 6-bit code u in 0..63 per byte; u ^ 32 with bit 5 copied into bits 6, 7
    // is u - 32 as a two's-complement byte
    const uint32_t u = ((lo[i] >> sl) & 0x0F0F0F0Fu) | (((hi[i] >> sh) & 0x03030303u) << 4);
    const uint32_t x = u ^ 0x20202020u, sg = x & 0x20202020u;
    w[i] = (int)(x | (sg << 1) | (sg << 2));
  }
  const uint32_t scw = lds16(sb + 192 + 2 * j);
  s0 = (float)(int8_t)(scw & 0xFFu);
  s1 = (float)(int8_t)(scw >> 8);
  d = f16_bits_to_f32(lds16(sb + 208));
}

// Integer dots of the two 16-value halves of a decoded sub-block of signed
// bytes (Q6_K, or NVFP4 through nvfp4_signed).
__device__ __forceinline__ void int_dots_halves(const int (&w)[8], const int (&q)[8], int& d0, int& d1) {
  int a0 = 0, a1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a0 = __dp4a(w[i], q[i], a0);
    a1 = __dp4a(w[i + 4], q[i + 4], a1);
  }
  d0 = a0;
  d1 = a1;
}

// ------------------------------------------------------------------ Q4_0

// Block b of a Q4_0 row (18-byte blocks, 2-byte aligned): the unsigned codes
// q (0..15) as int8x4 words in value order, and d.  The offset -8 is applied
// by the caller through the activation block's exact code sum.
__device__ __forceinline__ void q4_0_decode(const uint8_t* row, int b, int (&w)[8], float& d) {
  const uint8_t* blk = row + 18 * b;
  d = f16_bits_to_f32(lds16(blk));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = lds16(blk + 2 + 4 * i) | ((uint32_t)lds16(blk + 4 + 4 * i) << 16);
    w[i] = (int)(c & 0x0F0F0F0Fu);
    w[i + 4] = (int)((c >> 4) & 0x0F0F0F0Fu);
  }
}

// ------------------------------------------------------------------ Q4_1, Q5_0, Q5_1, MXFP4

// Bits 0..3 of x to bit 4 of bytes 0..3 (the fifth code bit of four values):
// the multiply places copies of x at bits 0, 7, 14 and 21, which do not
// overlap, so bit k lands at bit 8k with no carries.
__device__ __forceinline__ uint32_t q5_spread(uint32_t x) {
  return (((x & 15u) * 0x00204081u) & 0x01010101u) << 4;
}

// Block b of a Q4_1 row (20-byte blocks, 4-byte aligned): unsigned codes,
// d and m.
__device__ __forceinline__ void q4_1_decode(const uint8_t* row, int b, int (&w)[8], float& d, float& m) {
  const uint8_t* blk = row + 20 * b;
  const uint32_t dm = lds32(blk);
  d = f16_bits_to_f32(dm & 0xFFFFu);
  m = f16_bits_to_f32(dm >> 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = lds32(blk + 4 + 4 * i);
    w[i] = (int)(c & 0x0F0F0F0Fu);
    w[i + 4] = (int)((c >> 4) & 0x0F0F0F0Fu);
  }
}

// Block b of a Q5_0 row (22-byte blocks, 2-byte aligned): unsigned 5-bit
// codes (the offset -16 goes through the activation's code sum) and d.
__device__ __forceinline__ void q5_0_decode(const uint8_t* row, int b, int (&w)[8], float& d) {
  const uint8_t* blk = row + 22 * b;
  d = f16_bits_to_f32(lds16(blk));
  const uint32_t qh = lds16(blk + 2) | ((uint32_t)lds16(blk + 4) << 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = lds16(blk + 6 + 4 * i) | ((uint32_t)lds16(blk + 8 + 4 * i) << 16);
    w[i] = (int)((c & 0x0F0F0F0Fu) | q5_spread(qh >> (4 * i)));
    w[i + 4] = (int)(((c >> 4) & 0x0F0F0F0Fu) | q5_spread(qh >> (16 + 4 * i)));
  }
}

// Block b of a Q5_1 row (24-byte blocks, 8-byte aligned): unsigned 5-bit
// codes, d and m.
__device__ __forceinline__ void q5_1_decode(const uint8_t* row, int b, int (&w)[8], float& d, float& m) {
  const uint8_t* blk = row + 24 * b;
  const uint32_t dm = lds32(blk), qh = lds32(blk + 4);
  d = f16_bits_to_f32(dm & 0xFFFFu);
  m = f16_bits_to_f32(dm >> 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = lds32(blk + 8 + 4 * i);
    w[i] = (int)((c & 0x0F0F0F0Fu) | q5_spread(qh >> (4 * i)));
    w[i + 4] = (int)(((c >> 4) & 0x0F0F0F0Fu) | q5_spread(qh >> (16 + 4 * i)));
  }
}

// Four 4-bit codes (one per byte, 0..15) as signed bytes 2*E2M1(code): the
// codes packed as a 16-bit prmt selector, then the sign-split lookup of
// nvfp4_words made signed as in nvfp4_signed.
__device__ __forceinline__ uint32_t e2m1x4_signed(uint32_t codes) {
  const uint32_t t = codes | (codes >> 4);
  const uint32_t sel = (t & 0xFFu) | ((t >> 8) & 0xFF00u);
  const uint32_t pos = prmt(kE2M1x2Lo, kE2M1x2Hi, sel);
  const uint32_t neg = prmt(kE2M1x2Lo, kE2M1x2Hi, sel ^ 0x8888u);
  return pos | ((0x80808080u - neg) ^ 0x80808080u);
}

// Block b of an MXFP4 row (17-byte blocks, any alignment): the 32 values
// 2*E2M1(code) as signed int8x4 words in value order, and 2^(e - 127).  The
// block is read as five aligned words starting at or below it (up to 3
// bytes before and 3 bytes past its 17 bytes, inside the row's 4-byte
// rounded span) and realigned with funnel shifts.
__device__ __forceinline__ void mxfp4_decode(const uint8_t* row, int b, int (&w)[8], float& scale) {
  const uint8_t* blk = row + 17 * b;
  const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(blk) & 3u);
  const uint8_t* a = blk - mis;
  uint32_t r[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) r[i] = lds32(a + 4 * i);
  const uint32_t sh = 8u * mis;
  uint32_t v[5];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __funnelshift_r(r[i], r[i + 1], sh);
  v[4] = r[4] >> sh;
  const uint32_t e = v[0] & 0xFFu;
  scale = e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);   // 2^(e - 127)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = __funnelshift_r(v[i], v[i + 1], 8);   // code bytes 4i .. 4i+3
    w[i] = (int)e2m1x4_signed(c & 0x0F0F0F0Fu);
    w[i + 4] = (int)e2m1x4_signed((c >> 4) & 0x0F0F0F0Fu);
  }
}

// ------------------------------------------------------------------ BF16

// 8 bf16 values (16 bytes) -> fp32 (exact).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Values 8c .. 8c+7 of a float row in shared memory as fp32 (exact): BF16 and
// F16 rows hold 8 values in 16 bytes, F32 rows in 32.
template <int WT>
__device__ __forceinline__ void float_row_chunk8(const uint8_t* row, int c, float (&f)[8]) {
  if constexpr (WT == W_F32) {
    const float4 a = *reinterpret_cast<const float4*>(row + 32 * c);
    const float4 b = *reinterpret_cast<const float4*>(row + 32 * c + 16);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else if constexpr (WT == W_F16) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = f16_bits_to_f32(w[i] & 0xFFFFu);
      f[2 * i + 1] = f16_bits_to_f32(w[i] >> 16);
    }
  } else {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(row + 16 * c), f);
  }
}

}  // namespace qre
