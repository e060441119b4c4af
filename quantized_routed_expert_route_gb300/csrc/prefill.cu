// Prompt-path (prefill) kernels on the sm_103a tensor cores.
//
// One prompt chunk of T tokens through one routed-expert layer (Strata PR
// #292, "Summary/Pipeline": the prompt path runs the routed experts as
// grouped GEMMs, W4A4 with activations quantized to NVFP4 on the fly or W4A8
// with q8_1 activations; FreeToken PR #732, "Design", for the layer formula
// and the per-expert weight_scale_2 applied to each projection's fp32 output):
//
//   k_pf_count,   P1: the T*K routes sorted by expert (stable: route order
//   k_pf_scatter  t*K+k inside an expert), per-expert row offsets: per-block
//                 expert counts over slices of the routes, then every block
//                 places its slice after the earlier blocks' routes.
//   k_pf_quant    P2: every token's hidden state quantized once -- NVFP4 (per
//                 16 values: UE4M3 scale = amax/6 nearest-even, E2M1 codes
//                 nearest-even, global scale 1) or q8_1 -- and stored both as
//                 codes and as fp16 operands: the exact dequantized NVFP4
//                 values, or each q8_1 value q*d as an fp16 pair hi + lo.  The
//                 FP16 mode quantizes nothing: x rounded to fp16 is the operand.
//   k_pf_gemm<0>  P3: grouped gate_up GEMM.  A tile is (expert, 256 sorted
//                 rows, 128 intermediate columns): 128 gate rows and 128 up
//                 rows of the expert's NVFP4 bank are expanded to fp16
//                 (code * UE4M3 scale, exact) into swizzled shared-memory
//                 tiles, the rows' activations are gathered beside them, and
//                 one thread issues tcgen05 kind::f16 MMAs into two 128x256
//                 fp32 accumulators in tensor memory.  The epilogue applies
//                 s_gate / s_up and the GLU in fp32, requantizes each 16 (or
//                 32) intermediate values to NVFP4 (or q8_1), and stores the
//                 exact fp16 dequantized values (the FP16 mode stores the
//                 intermediate rounded to fp16).
//   k_pf_gemm<1>  P4: grouped down GEMM, (expert, 256 rows, 256 outputs)
//                 tiles over the requantized intermediate; the epilogue scales
//                 by s_down * routing weight and stores fp32 per route.
//   k_pf_combine  P6: out[t] = bf16(sum over k = 0..K-1 of the route rows),
//                 in route order, no atomics.
//
// W4A4 on a bank with the grouped TMA maps runs on the block-scaled FP4
// tensor cores instead (no fp16 operands): k_pf4_quant (a warp per token) also
// writes x's NVFP4 rows in sorted order and zeroes the fp32 token sums;
// k_pf4_gate_up (P3, 128 x 256 MMAs) and k_pf4_down (P4, 128 x 128 MMAs) are
// tcgen05 kind::mxf4nvf4 GEMMs, the second adding each route's scaled row
// into its token's sum by bulk reductions at L2 (P6 in completion order);
// k_pf4_finish rounds the sums to bf16.  The fixed-order
// mode stores each route's row instead and k_pf4_combine sums k = 0..K-1.
//
// Every product in the MMAs is of two exact fp16 values (NVFP4 code * scale,
// or a q8_1 value rounded to fp16 once), accumulated in fp32.
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "tc.cuh"

namespace qre {

// ------------------------------------------------------------------ tensor-core check

// D[128][N] = A[128][K] * B[N][K]^T, fp16 inputs (row-major), fp32 out, on
// the tensor cores: one CTA of 4 warps stages 64-wide K slices of A and B
// into swizzled shared-memory tiles, one thread issues four kind::f16 MMAs
// per slice into tensor memory, the warps read their 32 lanes back.
__global__ void __launch_bounds__(128, 1) k_tc_gemm_check(const uint16_t* A, const uint16_t* B, int K, int N,
                                                           float* D, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sa = base;
  uint8_t* sb = base + 16384;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = tc::idesc_f16(128, (uint32_t)N, false);
  uint32_t phase = 0;
  bool ok = true;
  for (int k0 = 0; k0 < K; k0 += 64) {
    for (int i = tid; i < 128 * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(sa + tc::sw128_chunk(r, c)) =
          *reinterpret_cast<const uint4*>(A + (size_t)r * K + k0 + 8 * c);
    }
    for (int i = tid; i < N * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(sb + tc::sw128_chunk(r, c)) =
          *reinterpret_cast<const uint4*>(B + (size_t)r * K + k0 + 8 * c);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_f16(tmem, tc::desc_sw128(smem_addr(sa) + 32 * kk), tc::desc_sw128(smem_addr(sb) + 32 * kk), idesc,
                    (k0 > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&bar);
    }
    if (!mbar_wait_bounded(&bar, phase, kWaitLimit)) ok = false;
    phase ^= 1u;
    tc::fence_after_sync();
  }
  for (int j0 = 0; j0 < N; j0 += 32) {
    uint32_t r[32];
    tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)j0, r);
    tc::tmem_ld_wait();
    const int m = 32 * warp + (tid & 31);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j0 + j < N) D[(size_t)m * N + j0 + j] = __uint_as_float(r[j]);
  }
  if (!ok) atomicOr(err, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_tc_gemm_check(const uint16_t* A, const uint16_t* B, int K, int N, float* D, int* err,
                                 cudaStream_t stream) {
  const size_t smem = 1024 + 16384 + (size_t)N * 128;
  cudaError_t e = cudaFuncSetAttribute(k_tc_gemm_check, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_tc_gemm_check<<<1, 128, smem, stream>>>(A, B, K, N, D, err);
  return cudaGetLastError();
}

// Block-scaled FP4 check: D[128, N] = sum over K of (A * sA) * (B * sB)^T
// with A [128][K/2] and B [N][K/2] packed E2M1 codes (value 2i in the low
// nibble of byte i) and sA [128][K/16], sB [N][K/16] UE4M3 scales, on the
// tcgen05 kind::mxf4nvf4 MMA: each 256-value K chunk's codes go to 128-byte
// swizzled tiles; for each of its four MMAs (64 values) the scales of each
// 128 rows go to a 512-byte atom (line r: the four scales of rows r, r+32,
// r+64, r+96) that tcgen05.cp copies to four tensor-memory columns; for
// N > 128 the scales of B rows 128..255 take the next four columns (eight a
// MMA).  N <= 256, a multiple of 16; rows of B (and their scales) beyond N
// read as zero.  Global loads check their alignment (a misaligned one is
// skipped and flags bit 1 of *err).
__global__ void __launch_bounds__(128, 1) k_fp4_gemm_check(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                                           const uint8_t* sB, int K, int N, float* D, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sa = base;                 // 128 rows x 128 bytes, swizzled
  uint8_t* sb = base + 16384;         // 256 rows x 128 bytes, swizzled
  uint8_t* ssa = base + 49152;        // four 512-byte scale atoms (one per MMA)
  uint8_t* ssb = base + 49152 + 2048; // eight: B rows 0..127, then 128..255
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int nbh = N > 128 ? 2 : 1;                          // 128-row halves of B
  const uint32_t t_sfa = tmem + 256, t_sfb = tmem + 272;    // 4 MMAs x 4 (A) and 4 x 4 * nbh (B) columns
  const uint32_t idesc = tc::idesc_mxf4nvf4(128, (uint32_t)N);
  const size_t rb = (size_t)K / 2, sb_row = (size_t)K / 16;
  uint32_t phase = 0;
  bool ok = true, misaligned = false;
  for (int k0 = 0; k0 < K; k0 += 256) {
    for (int i = tid; i < 256 * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      if (r < 128) {
        const uint8_t* pa = A + (size_t)r * rb + k0 / 2 + 16 * c;
        uint4 va = make_uint4(0, 0, 0, 0);
        if ((reinterpret_cast<uintptr_t>(pa) & 15) == 0) va = *reinterpret_cast<const uint4*>(pa);
        else misaligned = true;
        *reinterpret_cast<uint4*>(sa + tc::sw128_chunk(r, c)) = va;
      }
      const uint8_t* pb = B + (size_t)r * rb + k0 / 2 + 16 * c;
      uint4 vb = make_uint4(0, 0, 0, 0);
      if (r < N) {
        if ((reinterpret_cast<uintptr_t>(pb) & 15) == 0) vb = *reinterpret_cast<const uint4*>(pb);
        else misaligned = true;
      }
      *reinterpret_cast<uint4*>(sb + tc::sw128_chunk(r, c)) = vb;
    }
    // scale atoms: atom kk, line r (32), word c (4): rows r + 32 c, blocks 4 kk .. 4 kk + 3
    for (int i = tid; i < 4 * 32 * 4; i += 128) {
      const int kk = i >> 7, r = (i >> 2) & 31, c = i & 3;
      const int row = r + 32 * c;
      const uint8_t* qa = sA + (size_t)row * sb_row + k0 / 16 + 4 * kk;
      uint32_t wa = 0;
      if ((reinterpret_cast<uintptr_t>(qa) & 3) == 0) wa = *reinterpret_cast<const uint32_t*>(qa);
      else misaligned = true;
      *reinterpret_cast<uint32_t*>(ssa + 512 * kk + 16 * r + 4 * c) = wa;
      for (int hb = 0; hb < 2; ++hb) {
        const int brow = 128 * hb + row;
        const uint8_t* qb = sB + (size_t)brow * sb_row + k0 / 16 + 4 * kk;
        uint32_t wb = 0;
        if (brow < N) {
          if ((reinterpret_cast<uintptr_t>(qb) & 3) == 0) wb = *reinterpret_cast<const uint32_t*>(qb);
          else misaligned = true;
        }
        *reinterpret_cast<uint32_t*>(ssb + 2048 * hb + 512 * kk + 16 * r + 4 * c) = wb;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      for (int kk = 0; kk < 4; ++kk) {
        tc::tmem_cp_32x128b_x4(t_sfa + 4 * kk, tc::desc_plain(smem_addr(ssa + 512 * kk), 128));
        for (int hb = 0; hb < nbh; ++hb)
          tc::tmem_cp_32x128b_x4(t_sfb + 4 * nbh * kk + 4 * hb,
                                 tc::desc_plain(smem_addr(ssb + 2048 * hb + 512 * kk), 128));
      }
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_mxf4nvf4(tmem, tc::desc_sw128(smem_addr(sa) + 32 * kk), tc::desc_sw128(smem_addr(sb) + 32 * kk),
                         idesc, t_sfa + 4 * kk, t_sfb + 4 * nbh * kk, (k0 > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&bar);
    }
    if (!mbar_wait_bounded(&bar, phase, kWaitLimit)) ok = false;
    phase ^= 1u;
    tc::fence_after_sync();
  }
  for (int j0 = 0; j0 < N; j0 += 32) {
    uint32_t r[32];
    tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)j0, r);
    tc::tmem_ld_wait();
    const int m = 32 * warp + (tid & 31);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j0 + j < N) D[(size_t)m * N + j0 + j] = __uint_as_float(r[j]);
  }
  if (!ok) atomicOr(err, 1);
  if (misaligned) atomicOr(err, 2);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

cudaError_t launch_fp4_gemm_check(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, int K,
                                  int N, float* D, int* err, cudaStream_t stream) {
  const size_t smem = 1024 + 49152 + 2048 + 4096;
  cudaError_t e = cudaFuncSetAttribute(k_fp4_gemm_check, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_fp4_gemm_check<<<1, 128, smem, stream>>>(A, sA, B, sB, K, N, D, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ P1: routes sorted by expert

constexpr int kSortThreads = 1024;
constexpr int kSortRoutes = 1024;   // routes per block (the grid has at most kSortBlocks blocks)

// Blocks of the two sort passes for RT routes: block b takes the routes
// [b * per, (b + 1) * per), per = ceil(RT / blocks).
int pf_sort_blocks(long long RT) {
  const long long nb = (RT + kSortRoutes - 1) / kSortRoutes;
  return nb < 1 ? 1 : nb > kSortBlocks ? kSortBlocks : (int)nb;
}

// First pass: block b counts the valid routes of each expert in its slice
// (bcnt[b][e]).  Block 0 clears the error word (each prompt-path call starts
// clean; the second pass, a later launch, is the first to set it).
__global__ void __launch_bounds__(kSortThreads) k_pf_count(const __grid_constant__ PfParams p) {
  extern __shared__ int ssm[];
  int* cnt = ssm;   // [E]
  const int tid = threadIdx.x, b = blockIdx.x, E = p.E;
  if (b == 0 && tid == 0) *p.err = 0u;
  for (int e = tid; e < E; e += kSortThreads) cnt[e] = 0;
  __syncthreads();
  const int per = (p.RT + gridDim.x - 1) / gridDim.x;
  const int r0 = min(p.RT, b * per), r1 = min(p.RT, r0 + per);
  for (int r = r0 + tid; r < r1; r += kSortThreads) {
    const int e = __ldg(p.ids + r);
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kSortThreads) p.bcnt[(size_t)b * E + e] = cnt[e];
}

// Second pass: every block derives the experts' offsets (an exclusive scan of
// the per-expert totals; block 0 stores them) and its own first row of each
// expert (the offset plus the earlier blocks' counts), then places its slice
// warp by warp (each warp a consecutive sub-slice, its lanes ranked by
// __match_any_sync), so the order inside an expert is the route order: the
// stable sort.  Routes whose id is outside [0, E) are left out and flag the
// error word.
__global__ void __launch_bounds__(kSortThreads) k_pf_scatter(const __grid_constant__ PfParams p) {
  extern __shared__ int ssm[];
  constexpr int NW = kSortThreads / 32;
  const int E = p.E, tid = threadIdx.x, lane = tid & 31, w = tid >> 5, b = blockIdx.x;
  int* cnt = ssm;              // [NW][E]: per-warp counts, then each warp's first row of each expert
  int* base = cnt + NW * E;    // [E]
  int* pre = base + E;         // [E]
  int* wsum = pre + E;         // [33]
  for (int e = tid; e < E; e += kSortThreads) {
    int tot = 0, before = 0;
    for (int bb = 0; bb < (int)gridDim.x; ++bb) {
      const int c = p.bcnt[(size_t)bb * E + e];
      tot += c;
      if (bb < b) before += c;
    }
    base[e] = tot;
    pre[e] = before;
  }
  for (int i = tid; i < NW * E; i += kSortThreads) cnt[i] = 0;
  __syncthreads();
  const int total = block_exclusive_scan(base, E, wsum);
  if (b == 0) {
    for (int e = tid; e < E; e += kSortThreads) p.off[e] = base[e];
    if (tid == 0) p.off[E] = total;
  }
  const int per = (p.RT + gridDim.x - 1) / gridDim.x;
  const int s0 = min(p.RT, b * per), s1 = min(p.RT, s0 + per);
  const int wper = (s1 - s0 + NW - 1) / NW;
  const int r0 = min(s1, s0 + w * wper), r1 = min(s1, r0 + wper);
  bool bad = false;
  for (int r = r0 + lane; r < r1; r += 32) {
    const int e = __ldg(p.ids + r);
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[w * E + e], 1);
    } else {
      bad = true;
      if (p.inv) p.inv[r] = -1;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kSortThreads) {
    int acc = base[e] + pre[e];
    for (int ww = 0; ww < NW; ++ww) {
      const int c = cnt[ww * E + e];
      cnt[ww * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  for (int rb = r0; rb < r1; rb += 32) {
    const int r = rb + lane;
    const int e = (r < r1) ? __ldg(p.ids + r) : -1;
    const bool v = r < r1 && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (v) {
      p.perm[cnt[w * E + e] + rank] = r;
      if (p.inv) p.inv[r] = cnt[w * E + e] + rank;
    }
    __syncwarp();
    if (v && rank == 0) cnt[w * E + e] += __popc(peers);
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, kErrBadId);
}

size_t pf_count_smem(int E) { return sizeof(int) * (size_t)E; }
size_t pf_scatter_smem(int E) { return sizeof(int) * ((size_t)(kSortThreads / 32) * E + 2 * (size_t)E + 33); }

// ------------------------------------------------------------------ P2: activation quantizers

// E2M1 codes (nearest even, saturating) of v[i] / sv for eight values, as
// the IEEE fp32 division gives them: the codes of v * r (r = 1/sv rounded)
// are taken unless v * r lies within 2^-20 (relative) of an E2M1 rounding
// boundary -- the quotients differ by a few units in the last place, and
// the rounding is monotone, so equal codes at t(1 - 2^-20), t and
// t(1 + 2^-20) are the codes of the division -- else the division is done.
__device__ __forceinline__ uint32_t e2m1x8_div(const float* v, float sv, float r) {
  float t[8], tl[8], th[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    t[i] = v[i] * r;
    tl[i] = t[i] * 0.99999904632568359375f;   // 1 - 2^-20
    th[i] = t[i] * 1.00000095367431640625f;   // 1 + 2^-20
  }
  const uint32_t c = tc::e2m1x8_rne_sat(t);
  if (c == tc::e2m1x8_rne_sat(tl) && c == tc::e2m1x8_rne_sat(th)) return c;
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(v[i], sv);
  return tc::e2m1x8_rne_sat(q);
}

// NVFP4 quantization of 16 values (W4A4 activations and intermediate): the
// UE4M3 scale byte, the eight code bytes as two words, and the exact fp16
// dequantized values (code * scale) as eight f16x2 words.
__device__ __forceinline__ void nvfp4_quant16(const float* v, uint32_t& sbyte, uint32_t& c0, uint32_t& c1,
                                              uint32_t (&h)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  sbyte = tc::e4m3_rne_sat(__fdiv_rn(amax, 6.0f));
  const uint32_t s2 = tc::ue4m3x2_to_f16x2((uint16_t)(sbyte | (sbyte << 8)));   // (scale, scale)
  const float sv = f16_bits_to_f32(s2 & 0xFFFFu);
  if (sv > 0.f) {
    const float r = __frcp_rn(sv);
    c0 = e2m1x8_div(v, sv, r);
    c1 = e2m1x8_div(v + 8, sv, r);
  } else {
    c0 = c1 = 0u;
  }
  uint32_t a[4], b[4];
  tc::e2m1x8_to_f16x8(c0, a);
  tc::e2m1x8_to_f16x8(c1, b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = tc::hmul2(a[i], s2);
    h[4 + i] = tc::hmul2(b[i], s2);
  }
}

// q8_1 quantization of 32 values (W4A8 activations and intermediate, the same
// device function as the decode path): codes, d (fp16 value as fp32), and
// the fp16 values round(q * d) as sixteen f16x2 words.
__device__ __forceinline__ void q8_1_quant32_f16(const float (&v)[32], uint32_t (&qw)[8], float& dh, int& sum,
                                                 float& dfull, uint32_t (&h)[16]) {
  q8_1_quantize_block(v, qw, dfull, sum);
  dh = f16_bits_to_f32(f32_to_f16_bits_rn(dfull));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int q0 = (int)(int8_t)((qw[i >> 1] >> (16 * (i & 1))) & 0xFFu);
    const int q1 = (int)(int8_t)((qw[i >> 1] >> (16 * (i & 1) + 8)) & 0xFFu);
    const uint32_t lo = f32_to_f16_bits_rn((float)q0 * dh), hi = f32_to_f16_bits_rn((float)q1 * dh);
    h[i] = lo | (hi << 16);
  }
}

// W4A4 on the FP4 tensor cores: one warp per token.  Lane l quantizes the
// 16-value blocks l, l + 32, ... of the token (the rule of nvfp4_quant16),
// writes them to the token's row and to the sorted row of each of its valid
// routes (consecutive lanes: consecutive 8-byte code groups and scale bytes),
// and zeroes the token's fp32 sums when the route sum reduces into them.
__global__ void __launch_bounds__(256) k_pf4_quant(const __grid_constant__ PfParams p) {
  const int lane = threadIdx.x & 31;
  const int t = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (t >= p.T) return;
  const int nb = p.H / 16;
  const size_t rbx = (size_t)p.H / 2 + p.H / 16;
  const int myrow = lane < p.K ? __ldg(p.inv + (size_t)t * p.K + lane) : -1;
  for (int b0 = 0; b0 < nb; b0 += 32) {   // warp-uniform: the shuffles below need every lane
    const int b = b0 + lane;
    const bool on = b < nb;
    uint32_t sbyte = 0u, c0 = 0u, c1 = 0u;
    if (on) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H + 16 * b);
      float v[16];
      float f[8];
      bf16x8_to_f32(__ldg(src), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = f[i];
      bf16x8_to_f32(__ldg(src + 1), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 + i] = f[i];
      uint32_t h[8];
      nvfp4_quant16(v, sbyte, c0, c1, h);
      *reinterpret_cast<uint2*>(p.xq + (size_t)t * rbx + 8 * b) = make_uint2(c0, c1);
      p.xq[(size_t)t * rbx + p.H / 2 + b] = (uint8_t)sbyte;
    }
    for (int k = 0; k < p.K; ++k) {
      const int row = __shfl_sync(0xffffffffu, myrow, k);
      if (row < 0 || !on) continue;
      *reinterpret_cast<uint2*>(p.xs + (size_t)row * rbx + 8 * b) = make_uint2(c0, c1);
      p.xs[(size_t)row * rbx + p.H / 2 + b] = (uint8_t)sbyte;
    }
  }
  if (p.ysum) {
    float4* ys = reinterpret_cast<float4*>(p.ysum + (size_t)t * p.H);
    for (int i = lane; i < p.H / 4; i += 32) ys[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// One thread per 16 (W4A4) or 32 (W4A8, FP16) values of x.
__global__ void k_pf_quant(const __grid_constant__ PfParams p) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (p.mode == PF_FP16) {
    const int nb = p.H / 32;
    if (idx >= (long long)p.T * nb) return;
    const int t = (int)(idx / nb), b = (int)(idx - (long long)t * nb);
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H + 32 * b);
    uint4* dst = reinterpret_cast<uint4*>(p.x16 + (size_t)t * p.H + 32 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[8];
      bf16x8_to_f32(__ldg(src + i), f);
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = f32_to_f16_bits_rn(f[2 * j]) | (f32_to_f16_bits_rn(f[2 * j + 1]) << 16);
      dst[i] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    return;
  }
  if (p.mode == PF_W4A4) {
    const int nb = p.H / 16;
    if (idx >= (long long)p.T * nb) return;
    const int t = (int)(idx / nb), b = (int)(idx - (long long)t * nb);
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H + 16 * b);
    float v[16];
    {
      float f[8];
      bf16x8_to_f32(__ldg(src), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = f[i];
      bf16x8_to_f32(__ldg(src + 1), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 + i] = f[i];
    }
    uint32_t sbyte, c0, c1, h[8];
    nvfp4_quant16(v, sbyte, c0, c1, h);
    const size_t rbx = (size_t)p.H / 2 + p.H / 16;
    *reinterpret_cast<uint2*>(p.xq + (size_t)t * rbx + 8 * b) = make_uint2(c0, c1);
    p.xq[(size_t)t * rbx + p.H / 2 + b] = (uint8_t)sbyte;
    if (p.x16) {   // the fp16 operand of the kind::f16 GEMMs (not used on the FP4 tensor cores)
      uint4* dst = reinterpret_cast<uint4*>(p.x16 + (size_t)t * p.H + 16 * b);
      dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
      dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  } else {
    const int nb = p.H / 32;
    if (idx >= (long long)p.T * nb) return;
    const int t = (int)(idx / nb), b = (int)(idx - (long long)t * nb);
    float v[32];
    load_block32<true>(p.x + (size_t)t * p.H, b, v);
    uint32_t qw[8], h[16];
    float dh, dfull;
    int sum;
    q8_1_quant32_f16(v, qw, dh, sum, dfull, h);
    uint32_t* blk = reinterpret_cast<uint32_t*>(p.xq + ((size_t)t * nb + b) * 36);
    blk[0] = f32_to_f16_bits_rn(dfull) | (f32_to_f16_bits_rn(dfull * (float)sum) << 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) blk[1 + i] = qw[i];
    uint4* dst = reinterpret_cast<uint4*>(p.x16 + (size_t)t * p.H + 32 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    // the remainder q*d - fp16(q*d), also in fp16: hi + lo carries q*d to
    // about 2^-22, so the gate_up products see the q8_1 values themselves
    uint32_t l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q0 = (int)(int8_t)((qw[i >> 1] >> (16 * (i & 1))) & 0xFFu);
      const int q1 = (int)(int8_t)((qw[i >> 1] >> (16 * (i & 1) + 8)) & 0xFFu);
      const float p0 = (float)q0 * dh, p1 = (float)q1 * dh;   // exact
      const float r0 = p0 - f16_bits_to_f32(h[i] & 0xFFFFu), r1 = p1 - f16_bits_to_f32(h[i] >> 16);
      l[i] = f32_to_f16_bits_rn(r0) | (f32_to_f16_bits_rn(r1) << 16);
    }
    uint4* dlo = reinterpret_cast<uint4*>(p.x16lo + (size_t)t * p.H + 32 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) dlo[i] = make_uint4(l[4 * i], l[4 * i + 1], l[4 * i + 2], l[4 * i + 3]);
  }
}

// ------------------------------------------------------------------ P3 / P4: grouped GEMMs

constexpr int kPfThreads = 512;     // 16 warps: all stage operands, one thread issues MMAs, all run the epilogue
constexpr int kPfTileRows = 256;
constexpr int kPfMaxStages = 3;
constexpr uint64_t kSpinLimit = 2000000000ull;   // an MMA-barrier wait gives up after 2 s of device time
constexpr int kPfBRawBytes = 9216;  // raw NVFP4 of 256 weight rows x 64 values: 32 code bytes + 4 scale bytes each

// Shared-memory plan of the GEMM (1024-byte aligned base):
//   A stages  [NS][A rows 0..127 | A rows 128..255 (| low parts, SPLIT)]
//   B16       [2][256 rows x 64 fp16, swizzled]         (the MMA's B operand)
//   Braw      [NS][256 x 32 code bytes | 256 x 4 scale bytes]
// A and Braw of chunk c + NS - 1 are copied (cp.async) while chunk c is
// expanded and multiplied.
template <bool SPLIT>
struct PfPlan {
  static constexpr int kStages = SPLIT ? 2 : 3;
  static constexpr int kABytes = SPLIT ? 65536 : 32768;
  static constexpr int kB16Off = kStages * kABytes;
  static constexpr int kBRawOff = kB16Off + 2 * 32768;
  static constexpr int kBytes = kBRawOff + kStages * kPfBRawBytes;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Issue the copies of K chunk kc of the current tile into A stage / Braw stage.
template <int PHASE, bool SPLIT>
__device__ __forceinline__ void pf_prefetch(const PfParams& p, const int* arow, const uint8_t* brp, int kc, int Kd,
                                            uint8_t* astage, uint8_t* braw, int tid) {
  const uint16_t* asrc = PHASE == 0 ? p.x16 : p.i16;
  const int k0 = kc * 64;
  constexpr int NA = SPLIT ? 8 : 4;
#pragma unroll
  for (int j = 0; j < NA; ++j) {
    const int i = tid + (j & 3) * kPfThreads;
    const int m = i >> 3, c = i & 7;
    const int src = arow[m];
    const uint16_t* as = (j < 4) ? asrc : p.x16lo;
    const uint16_t* g = as + (size_t)(src >= 0 ? src : 0) * Kd + k0 + 8 * c;
    cp_async16(smem_addr(astage + (j < 4 ? 0 : 32768) + (m < 128 ? 0 : 16384) + tc::sw128_chunk(m & 127, c)), g,
               src >= 0);
  }
  const int brow = tid >> 1, bh = tid & 1;
  cp_async16(smem_addr(braw + brow * 32 + 16 * bh), brp + (k0 + 32 * bh) / 2, true);
  if (bh == 0) cp_async4(smem_addr(braw + 8192 + brow * 4), brp + Kd / 2 + k0 / 16);
}

// PHASE 0: gate_up (K = H; B rows = 128 gate + 128 up rows; epilogue GLU +
// requant); PHASE 1: down (K = I; B rows = 256 output rows; epilogue scales).
// SPLIT (W4A8 gate_up): the activations are the fp16 pair hi + lo and each
// product is formed as hi*B + lo*B into the same accumulator.
template <int PHASE, bool SPLIT>
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(const __grid_constant__ PfParams p) {
  using Plan = PfPlan<SPLIT>;
  constexpr int NS = Plan::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t mma_bar[kPfMaxStages];
  __shared__ uint32_t tmem_base;
  __shared__ int tile_pre[kMaxE + 1];
  __shared__ int wsum[33];
  __shared__ int arow[kPfTileRows];
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const int NT = PHASE == 0 ? p.I / 128 : p.H / 256;   // column tiles per expert
  const int Kd = PHASE == 0 ? p.H : p.I;               // reduction length
  const int nK = Kd / 64;
  for (int e = tid; e < E; e += kPfThreads) {
    const int M = p.off[e + 1] - p.off[e];
    tile_pre[e] = ((M + kPfTileRows - 1) / kPfTileRows) * NT;
  }
  __syncthreads();
  const int total = block_exclusive_scan(tile_pre, E, wsum);
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&mma_bar[s], 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = tc::idesc_f16(128, 256, false);
  uint32_t chunk = 0;   // chunks multiplied so far (all tiles): picks the stage and barrier phase
  bool ok = true;
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    // the expert of tile t: the largest e with tile_pre[e] <= t (never an empty one)
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_pre[mid] <= t) lo = mid;
      else hi = mid;
    }
    const int e = lo;
    const int tl = t - tile_pre[e];
    const int Me = p.off[e + 1] - p.off[e];
    const int mtiles = (Me + kPfTileRows - 1) / kPfTileRows;
    const int mt = tl % mtiles, nt = tl / mtiles;
    const int rows = min(kPfTileRows, Me - mt * kPfTileRows);
    const int srow0 = p.off[e] + mt * kPfTileRows;
    for (int m = tid; m < kPfTileRows; m += kPfThreads)
      arow[m] = (m < rows) ? (PHASE == 0 ? p.perm[srow0 + m] / p.K : srow0 + m) : -1;
    __syncthreads();   // arow visible; the previous tile's epilogue is done with tensor memory
    tc::fence_after_sync();
    const int rb = PHASE == 0 ? p.rb_gu : p.rb_dn;
    const int brow = tid >> 1, bh = tid & 1;
    const size_t bsrc_row = PHASE == 0 ? ((size_t)e * 2 * p.I + (brow < 128 ? nt * 128 + brow : p.I + nt * 128 + brow - 128))
                                       : ((size_t)e * p.H + (size_t)nt * 256 + brow);
    const uint8_t* brp = (PHASE == 0 ? p.gu_bank : p.dn_bank) + bsrc_row * rb;
    // prologue: chunks 0 .. NS-2 in flight (their stages were last read by
    // MMAs this thread already waited for at the end of the previous tile)
#pragma unroll
    for (int j = 0; j < NS - 1; ++j) {
      if (j < nK) {
        const uint32_t s = (chunk + j) % NS;
        pf_prefetch<PHASE, SPLIT>(p, arow, brp, j, Kd, base + s * Plan::kABytes,
                                  base + Plan::kBRawOff + s * kPfBRawBytes, tid);
      }
      cp_async_commit();
    }
    for (int kc = 0; kc < nK; ++kc, ++chunk) {
      const uint32_t s = chunk % NS;
      uint8_t* ast = base + s * Plan::kABytes;
      const uint8_t* braw = base + Plan::kBRawOff + s * kPfBRawBytes;
      uint8_t* b16 = base + Plan::kB16Off + (chunk & 1u) * 32768;
      cp_async_wait<NS - 2>();   // this thread's copies of chunk kc have landed
      fence_proxy_async_smem();
      __syncthreads();           // everyone's copies of chunk kc are visible; MMA(chunk - 2) is done (see below)
      {
        // expand this thread's 32 NVFP4 weight values to fp16 (code * scale, exact)
        const uint4 cw = *reinterpret_cast<const uint4*>(braw + brow * 32 + 16 * bh);
        const uint16_t sw = *reinterpret_cast<const uint16_t*>(braw + 8192 + brow * 4 + 2 * bh);
        const uint32_t s2 = tc::ue4m3x2_to_f16x2(sw);
        const uint32_t s0 = prmt(s2, 0u, 0x1010u), s1 = prmt(s2, 0u, 0x3232u);
        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t h[4];
          tc::e2m1x8_to_f16x8(cws[q], h);
          const uint32_t sc = q < 2 ? s0 : s1;
          *reinterpret_cast<uint4*>(b16 + tc::sw128_chunk(brow, 4 * bh + q)) =
              make_uint4(tc::hmul2(h[0], sc), tc::hmul2(h[1], sc), tc::hmul2(h[2], sc), tc::hmul2(h[3], sc));
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
        const uint32_t a0 = smem_addr(ast), a1 = a0 + 16384, b0 = smem_addr(b16);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
          const uint64_t bd = tc::desc_sw128(b0 + 32 * kk);
          tc::mma_f16(tmem, tc::desc_sw128(a0 + 32 * kk), bd, idesc, acc);
          if (SPLIT) tc::mma_f16(tmem, tc::desc_sw128(a0 + 32768 + 32 * kk), bd, idesc, 1u);
          if (rows > 128) {
            tc::mma_f16(tmem + 256, tc::desc_sw128(a1 + 32 * kk), bd, idesc, acc);
            if (SPLIT) tc::mma_f16(tmem + 256, tc::desc_sw128(a1 + 32768 + 32 * kk), bd, idesc, 1u);
          }
        }
        tc::mma_commit(&mma_bar[s]);
      }
      // Chunk kc + NS - 1 goes to the stage that MMA(chunk - 1) read: wait for
      // it (this also covers the B16 buffer that chunk + 1 will overwrite).
      if (chunk >= 1) {
        const uint32_t pc = chunk - 1;
        if (!mbar_wait_spin(&mma_bar[pc % NS], (pc / NS) & 1u, kSpinLimit)) ok = false;
      }
      if (kc + NS - 1 < nK) {
        const uint32_t s2 = (chunk + NS - 1) % NS;
        pf_prefetch<PHASE, SPLIT>(p, arow, brp, kc + NS - 1, Kd, base + s2 * Plan::kABytes,
                                  base + Plan::kBRawOff + s2 * kPfBRawBytes, tid);
      }
      cp_async_commit();
    }
    {
      const uint32_t last = chunk - 1;
      if (!mbar_wait_spin(&mma_bar[last % NS], (last / NS) & 1u, kSpinLimit)) ok = false;
    }
    tc::fence_after_sync();
    // epilogue: warp w reads lanes 32*(w%4).. of each accumulator, column group w/4
    const int q = warp & 3, cg = warp >> 2;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    for (int h = 0; h < 2; ++h) {
      if (h == 1 && rows <= 128) break;
      const int m = h * 128 + 32 * q + lane;
      const bool valid = m < rows;
      if (PHASE == 0) {
        const float sg = __ldg(p.scales + 4 * e + 0), su = __ldg(p.scales + 4 * e + 1);
        float a[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t g16[16], u16[16];
          tc::tmem_ld16(tq + h * 256 + 32 * cg + 16 * half, g16);
          tc::tmem_ld16(tq + h * 256 + 128 + 32 * cg + 16 * half, u16);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            a[16 * half + j] = glu_act(__uint_as_float(g16[j]) * sg, __uint_as_float(u16[j]) * su, p.glu);
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.i16 + (size_t)(srow0 + m) * p.I + nt * 128 + 32 * cg);
          if (p.mode == PF_FP16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t hw[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                hw[j] = f32_to_f16_bits_rn(a[8 * i + 2 * j]) | (f32_to_f16_bits_rn(a[8 * i + 2 * j + 1]) << 16);
              dst[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
          } else if (p.mode == PF_W4A4) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              uint32_t sbyte, c0, c1, hw[8];
              nvfp4_quant16(a + 16 * b, sbyte, c0, c1, hw);
              dst[2 * b] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              dst[2 * b + 1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            }
          } else {
            uint32_t qw[8], hw[16];
            float dh, dfull;
            int sum;
            q8_1_quant32_f16(a, qw, dh, sum, dfull, hw);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
          }
        }
      } else {
        const float sd = __ldg(p.scales + 4 * e + 2);
        const int r = valid ? p.perm[srow0 + m] : 0;
        const float f = valid ? sd * __ldg(p.w + r) : 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tc::tmem_ld32(tq + h * 256 + 64 * cg + 32 * cc, v);
          tc::tmem_ld_wait();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(p.y + (size_t)r * p.H + nt * 256 + 64 * cg + 32 * cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(v[4 * i]) * f, __uint_as_float(v[4 * i + 1]) * f,
                                   __uint_as_float(v[4 * i + 2]) * f, __uint_as_float(v[4 * i + 3]) * f);
          }
        }
      }
    }
    tc::fence_before_sync();
  }
  if (!ok) atomicOr(p.err, kErrTimeout);
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

size_t pf_gemm_smem() {
  constexpr int a = PfPlan<false>::kBytes, b = PfPlan<true>::kBytes;
  return 1024 + (size_t)(a > b ? a : b);
}

// ------------------------------------------------------------------ P6: fixed-order combine

// out[t][n] = bf16(sum over k = 0..K-1 of y[t*K+k][n]), valid routes only.
__global__ void k_pf_combine(const __grid_constant__ PfParams p) {
  route_sum4(p.ids, p.y, p.out, p.T, p.K, p.E, p.H, (long long)blockIdx.x * blockDim.x + threadIdx.x);
}

// ------------------------------------------------------------------ W4A4 on the FP4 tensor cores

namespace {

constexpr int kF4Threads = 448;    // warp 0 TMA, warp 1 MMA, warps 2-5 scales, warps 6..13 epilogue
constexpr int kF4Code = 16384;     // one operand's codes per stage: 128 rows x 128 bytes (256 values)
constexpr int kF4Scale = 2048;     // its scales: 128 rows x 16 bytes
constexpr int kF4Op = kF4Code + kF4Scale;
constexpr int kF4Stage = 2 * kF4Op;     // the activation rows' operand, then the weight rows'
constexpr int kF4EpRow = 528;           // down epilogue: one row's 128 fp32 outputs, padded to spread banks

constexpr int kF4DownStages = 4;       // down stages; tensor memory: 256 accumulator + 4 * 32 scale columns

// 2-D TMA load of one box at (x, y) with an L2 cache policy (the activation
// rows and the token sums evict last, the weights normally: a weight tile is
// read again by the expert's other row blocks soon after).
__device__ __forceinline__ void f4_tma(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// out[0 .. bytes/4) += the fp32 values at src, as one asynchronous bulk
// reduction performed at L2 (16-byte aligned addresses, bytes a multiple of
// 16), with an L2 cache policy for the destination lines.
__device__ __forceinline__ void bulk_reduce_add_f32(float* out, const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.L2::cache_hint.add.f32 [%0], [%1], %2, %3;"
               ::"l"(out), "r"(smem_addr(src)), "r"(bytes), "l"(pol) : "memory");
}
// out[0 .. bytes) = the bytes at src, as one asynchronous bulk copy (the same alignment rules).
__device__ __forceinline__ void bulk_store(void* out, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(out), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk operations have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and are complete
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bounded wait (2 s of device time) that also gives up once another role of
// the CTA has.
// With `sleepy`, the waiting warp pauses between polls (roles off the
// critical path, so that they leave issue slots to the others).
__device__ __forceinline__ bool f4_wait(uint64_t* bar, uint32_t parity, volatile int* abort, bool sleepy = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (sleepy) __nanosleep(128);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kSpinLimit) {
        *abort = 1;
        return false;
      }
    }
  }
}

// One lane quarter of a stage's MMA scales in tensor memory (the warp with
// that quarter, q = warp % 4): the scale tile of one operand holds, for each
// of 128 rows R, 16 UE4M3 scales (four per MMA kk, K order); column 4 kk + c
// of every lane l of every quarter holds the four scales of row (l % 32) +
// 32 c for MMA kk -- the block-scaled MMA's layout for 128 rows, replicated in
// each quarter.  Lane l reads rows l, l + 32, l + 64, l + 96 (16 bytes each).
__device__ __forceinline__ void f4_scales_to_tmem(const uint8_t* tile, uint32_t taddr, int lane) {
  uint32_t col[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + 16 * (lane + 32 * c));
    col[c] = v.x;
    col[4 + c] = v.y;
    col[8 + c] = v.z;
    col[12 + c] = v.w;
  }
  tc::tmem_st16(taddr, col);
}

// Tile t of the sequence every role walks: row blocks of 128 sorted rows,
// expert by expert (rbpre: the prefix of each expert's row blocks), each
// with ncb column blocks.  The expert cursor only moves forward.
struct F4Tile {
  int e, row0, rows, cb;
};
__device__ __forceinline__ bool f4_tile(int t, int ncb, const int* rbpre, const int* soff, int E, int& ecur,
                                        F4Tile& tl) {
  const int rbg = t / ncb;
  if (rbg >= rbpre[E]) return false;
  while (rbpre[ecur + 1] <= rbg) ++ecur;
  tl.e = ecur;
  tl.row0 = soff[ecur] + 128 * (rbg - rbpre[ecur]);
  tl.rows = min(128, soff[ecur + 1] - tl.row0);
  tl.cb = t - rbg * ncb;
  return true;
}

}  // namespace

// Fixed-order route sum: out[t] = bf16(sum over k = 0..K-1 of the route rows), four values a thread.
__global__ void k_pf4_combine(const __grid_constant__ Pf4Params p) {
  route_sum4(p.ids, p.y, p.out, p.T, p.K, p.E, p.H, (long long)blockIdx.x * blockDim.x + threadIdx.x);
}

// out[t] = bf16 of the fp32 token sum (round to nearest even), four values a thread.
__global__ void k_pf4_finish(const __grid_constant__ Pf4Params p) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)p.T * (p.H / 4)) return;
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p.y) + i);
  uint2 o;
  o.x = f32_to_bf16_bits_rn(v.x) | (f32_to_bf16_bits_rn(v.y) << 16);
  o.y = f32_to_bf16_bits_rn(v.z) | (f32_to_bf16_bits_rn(v.w) << 16);
  reinterpret_cast<uint2*>(p.out)[i] = o;
}

// Grouped down GEMM of the W4A4 prompt path on tcgen05 kind::mxf4nvf4 (MMA
// M = N = 128, K = 64 per instruction): tile = (expert, 128 sorted rows, 128
// output rows), the rows' NVFP4 intermediate and the expert's NVFP4 down rows
// (codes and scales) by 2-D TMA, one 256-value chunk of I per stage.  The
// epilogue scales each route's row by s_down * w and adds it into its
// token's fp32 sum with bulk reductions at L2 (the route sum; see
// k_pf4_finish), or, with p.fixed, stores it as the route's own fp32 row for
// k_pf4_combine.
// Roles: warp 0 issues the TMA copies; warps 2..5 (one per tensor-memory
// lane quarter) store each stage's scales from its 128 x 16-byte scale tiles
// into tensor memory; warp 1 issues the MMAs; warps 6..9 (one per lane
// quarter, whole rows, so that each route row is one 512-byte reduction) run
// the epilogue; warps 10..13 have no role.
// The accumulators are double-buffered, so a tile's epilogue overlaps the
// next tile's MMAs.  One CTA per SM walks the tiles (blockIdx.x, +
// gridDim.x, ...).  Every product of two scaled E2M1 values is exact in
// fp32 and the MMA accumulates in fp32.
__global__ void __launch_bounds__(kF4Threads, 1) k_pf4_down(const __grid_constant__ Pf4Params p) {
  constexpr int NS = kF4DownStages;
  static_assert(256 + NS * 32 <= 512, "tensor memory: two 128-column accumulators and the stages' scales");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[NS], ready[NS], empty[NS], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = base;
  uint8_t* ep = base + NS * kF4Stage;                        // down: the epilogue rows
  int* soff = reinterpret_cast<int*>(ep + 128 * kF4EpRow);   // [E+1] first sorted row of each expert
  int* rbpre = soff + (p.E + 1);                             // [E+1] row blocks before each expert
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E;
  const int nchunk = p.I / 256;
  const int ncb = p.H / 128;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&ready[i], 4);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);   // the epilogue threads that read a buffer
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  for (int e = tid; e <= E; e += kF4Threads) soff[e] = p.off[e];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32, e0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
      if (e0 + i < E) local += (soff[e0 + i + 1] - soff[e0 + i] + 127) / 128;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i)
      if (e0 + i < E) {
        rbpre[e0 + i] = run;
        run += (soff[e0 + i + 1] - soff[e0 + i] + 127) / 128;
      }
    if (lane == 31) rbpre[E] = incl;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      const uint64_t pw = l2_policy_evict_normal(), pa = l2_policy_evict_last();
      int ecur = 0, q = 0;
      F4Tile tl;
      for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x) {
        const int yb = tl.e * p.H + 128 * tl.cb;   // the tile's first down row
        bool ok = true;
        for (int kc = 0; kc < nchunk; ++kc, ++q) {
          const int s = q % NS;
          if (q >= NS && !f4_wait(&empty[s], (uint32_t)(((q / NS) & 1) ^ 1), abort, true)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)s * kF4Stage;
          uint8_t* sb = st + kF4Op;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kF4Stage);
          f4_tma(st, &p.map_in, 128 * kc, tl.row0, &full[s], pa);
          f4_tma(st + kF4Code, &p.map_ins, p.I / 2 + 16 * kc, tl.row0, &full[s], pa);
          f4_tma(sb, &p.map_wdn, 128 * kc, yb, &full[s], pw);
          f4_tma(sb + kF4Code, &p.map_wdns, p.I / 2 + 16 * kc, yb, &full[s], pw);
        }
        if (!ok) break;
      }
      // wait (bounded) for the last copies issued (complete already unless a role gave up)
      for (int qn = q - NS < 0 ? 0 : q - NS; qn < q; ++qn)
        mbar_wait_spin(&full[qn % NS], (uint32_t)((qn / NS) & 1), kSpinLimit);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---- scales: this warp's lane quarter of both operands' scale columns
    const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256u;
    int ecur = 0, q = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x) {
      bool ok = true;
      for (int kc = 0; kc < nchunk; ++kc, ++q) {
        const int s = q % NS;
        if (!f4_wait(&full[s], (uint32_t)((q / NS) & 1), abort)) {
          ok = false;
          break;
        }
        const uint8_t* st = stages + (size_t)s * kF4Stage;
        f4_scales_to_tmem(st + kF4Code, tq + (uint32_t)(s * 32), lane);
        f4_scales_to_tmem(st + kF4Op + kF4Code, tq + (uint32_t)(s * 32 + 16), lane);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[s]);
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ---- tensor-memory scale copies and MMA issue
    const uint32_t idesc = tc::idesc_mxf4nvf4(128, 128);
    int ecur = 0, q = 0, ntile = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x, ++ntile) {
      const int buf = ntile & 1;
      if (ntile >= 2 && !f4_wait(&acc_empty[buf], (uint32_t)(((ntile >> 1) - 1) & 1), abort)) break;
      tc::fence_after_sync();
      bool ok = true;
      for (int kc = 0; kc < nchunk; ++kc, ++q) {
        const int s = q % NS;
        if (!f4_wait(&ready[s], (uint32_t)((q / NS) & 1), abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // the copies are complete (the scale warps saw it); this acquire
          // orders them for this thread's MMAs as well
          mbar_try_wait(&full[s], (uint32_t)((q / NS) & 1));
          tc::fence_after_sync();
          const uint32_t st = smem_addr(stages + (size_t)s * kF4Stage);
          const uint32_t sf = tmem + 256 + (uint32_t)(s * 32);   // the scale warps' columns of this stage
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_mxf4nvf4(tmem + 128 * buf, tc::desc_sw128(st + 32 * kk), tc::desc_sw128(st + kF4Op + 32 * kk), idesc,
                             sf + 4 * kk, sf + 16 + 4 * kk, (kc > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);   // the stage's smem and scale columns are free once these MMAs are done
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(&acc_full[buf]);
      __syncwarp();
    }
    if (lane == 0) {
      tc::mma_commit(&drain);   // everything this thread issued is complete before the dealloc
      mbar_wait_spin(&drain, 0u, kSpinLimit);
    }
  } else if (warp >= 6 && warp < 10) {
    // ---- epilogue: warp w reads tensor-memory lanes 32 * (w % 4) .. + 31, one tile row a thread
    const int qd = warp & 3;
    float* mine = reinterpret_cast<float*>(ep + (size_t)(32 * qd + lane) * kF4EpRow);   // down: this row's 128 outputs
    const uint64_t pkeep = l2_policy_evict_last();   // the token sums stay in L2 for k_pf4_finish
    int ecur = 0, ntile = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x, ++ntile) {
      const int buf = ntile & 1;
      if (!f4_wait(&acc_full[buf], (uint32_t)((ntile >> 1) & 1), abort, true)) break;
      tc::fence_after_sync();
      const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(128 * buf);
      const int m = 32 * qd + lane;
      const bool valid = m < tl.rows;
      const int row = tl.row0 + m;
      {
        const float sd = __ldg(p.scales + 4 * tl.e + 2);
        const int r = valid ? p.perm[row] : 0;
        const float f = valid ? sd * __ldg(p.w + r) : 0.f;
        bulk_wait_read();   // the previous tile's reduction has read this row
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          uint32_t v[32];
          tc::tmem_ld32(tq + 32 * j4, v);
          tc::tmem_ld_wait();
          if (j4 == 3) {
            tc::fence_before_sync();
            mbar_arrive(&acc_empty[buf]);
          }
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(mine + 32 * j4 + i) =
                make_float4(__uint_as_float(v[i]) * f, __uint_as_float(v[i + 1]) * f, __uint_as_float(v[i + 2]) * f,
                            __uint_as_float(v[i + 3]) * f);
        }
        if (valid) {
          fence_proxy_async_smem();
          if (p.fixed) bulk_store(p.y + (size_t)r * p.H + 128 * tl.cb, mine, 512);   // the route's own row
          else bulk_reduce_add_f32(p.y + (size_t)(r / p.K) * p.H + 128 * tl.cb, mine, 512, pkeep);
          bulk_commit();
        }
      }
    }
    bulk_wait_done();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && abort_flag) atomicOr(p.err, kErrTimeout);
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

size_t pf4_down_smem(int E) {
  return 1024 + (size_t)kF4DownStages * kF4Stage + 128 * kF4EpRow + 8 * ((size_t)E + 1);
}

// W4A4 gate_up with one N = 256 MMA per 64 values: the tile is (expert, 128
// sorted rows, 128 intermediate columns) -- the 128 gate rows then the 128
// up rows of the column block form one 256-row B operand, so each
// block-scaled MMA (M = 128, N = 256, K = 64) does twice the work of the
// 128-wide tile for about the same issue cost.  Tensor memory then holds a
// single 256-column accumulator (gate in columns 0..127, up in 128..255)
// beside the stages' scales (A: four columns an MMA; B: eight, rows 128..255
// in the second four), so the next tile's MMAs wait until the epilogue has
// read the accumulator; sixteen epilogue warps (four per lane quarter, two
// 16-value blocks each) keep that short.  Roles otherwise as k_pf4_gemm:
// warp 0 TMA, warp 1 MMA, warps 2..5 scales (one per lane quarter), warps
// 6..21 epilogue.
namespace {
constexpr int kGuThreads = 704;
constexpr int kGuStages = 4;
constexpr int kGuA = kF4Op;                       // 18,432: x rows' codes then scales
constexpr int kGuBCode = 2 * kF4Code;             // 32,768: 256 weight rows x 128 bytes
constexpr int kGuStage = kGuA + kGuBCode + 2 * kF4Scale;   // 55,296
constexpr int kGuSf = 48;                         // scale columns of a stage
static_assert(kGuStage % 1024 == 0 && kGuA % 1024 == 0, "1024-byte aligned code tiles");
static_assert(256 + kGuStages * kGuSf <= 512, "tensor memory: the accumulator and the stages' scales");

// One lane quarter of a stage's B scales (256 rows: gate rows then up rows,
// 16 bytes each) into its 32 columns: column 8 kk + 4 h + c of lane l holds
// the four scales of row 128 h + (l % 32) + 32 c for MMA kk.
__device__ __forceinline__ void gu_scales_b_to_tmem(const uint8_t* tile, uint32_t taddr, int lane) {
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + 2048 * h + 16 * (lane + 32 * c));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int col = 8 * kk + 4 * h + c;
        if (col < 16) lo[col] = w[kk];
        else hi[col - 16] = w[kk];
      }
    }
  tc::tmem_st16(taddr, lo);
  tc::tmem_st16(taddr + 16, hi);
}
}  // namespace

__global__ void __launch_bounds__(kGuThreads, 1) k_pf4_gate_up(const __grid_constant__ Pf4Params p) {
  constexpr int NS = kGuStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[NS], ready[NS], empty[NS], acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = base;
  int* soff = reinterpret_cast<int*>(base + NS * kGuStage);   // [E+1] first sorted row of each expert
  int* rbpre = soff + (p.E + 1);                               // [E+1] row blocks before each expert
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E;
  const int nchunk = p.H / 256;
  const int ncb = p.I / 128;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&ready[i], 4);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, 512);
    mbar_init(&drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  for (int e = tid; e <= E; e += kGuThreads) soff[e] = p.off[e];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32, e0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
      if (e0 + i < E) local += (soff[e0 + i + 1] - soff[e0 + i] + 127) / 128;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i)
      if (e0 + i < E) {
        rbpre[e0 + i] = run;
        run += (soff[e0 + i + 1] - soff[e0 + i] + 127) / 128;
      }
    if (lane == 31) rbpre[E] = incl;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      const uint64_t pw = l2_policy_evict_normal(), pa = l2_policy_evict_last();
      int ecur = 0, q = 0;
      F4Tile tl;
      for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x) {
        const int yb = tl.e * 2 * p.I + 128 * tl.cb;   // the tile's first gate row (its up rows are I further)
        bool ok = true;
        for (int kc = 0; kc < nchunk; ++kc, ++q) {
          const int s = q % NS;
          if (q >= NS && !f4_wait(&empty[s], (uint32_t)(((q / NS) & 1) ^ 1), abort, true)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)s * kGuStage;
          uint8_t* sb = st + kGuA;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kGuStage);
          f4_tma(st, &p.map_xs, 128 * kc, tl.row0, &full[s], pa);
          f4_tma(st + kF4Code, &p.map_xss, p.H / 2 + 16 * kc, tl.row0, &full[s], pa);
          f4_tma(sb, &p.map_wgu, 128 * kc, yb, &full[s], pw);
          f4_tma(sb + kF4Code, &p.map_wgu, 128 * kc, yb + p.I, &full[s], pw);
          f4_tma(sb + kGuBCode, &p.map_wgus, p.H / 2 + 16 * kc, yb, &full[s], pw);
          f4_tma(sb + kGuBCode + kF4Scale, &p.map_wgus, p.H / 2 + 16 * kc, yb + p.I, &full[s], pw);
        }
        if (!ok) break;
      }
      for (int qn = q - NS < 0 ? 0 : q - NS; qn < q; ++qn)
        mbar_wait_spin(&full[qn % NS], (uint32_t)((qn / NS) & 1), kSpinLimit);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---- scales: this warp's lane quarter of both operands' scale columns
    const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256u;
    int ecur = 0, q = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x) {
      bool ok = true;
      for (int kc = 0; kc < nchunk; ++kc, ++q) {
        const int s = q % NS;
        if (!f4_wait(&full[s], (uint32_t)((q / NS) & 1), abort)) {
          ok = false;
          break;
        }
        const uint8_t* st = stages + (size_t)s * kGuStage;
        f4_scales_to_tmem(st + kF4Code, tq + (uint32_t)(s * kGuSf), lane);
        gu_scales_b_to_tmem(st + kGuA + kGuBCode, tq + (uint32_t)(s * kGuSf + 16), lane);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[s]);
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ---- MMA issue: one 128 x 256 x 64 block-scaled MMA per 64 values
    const uint32_t idesc = tc::idesc_mxf4nvf4(128, 256);
    int ecur = 0, q = 0, ntile = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x, ++ntile) {
      // the single accumulator: the previous tile's epilogue has read it
      if (ntile >= 1 && !f4_wait(&acc_empty, (uint32_t)((ntile - 1) & 1), abort)) break;
      tc::fence_after_sync();
      bool ok = true;
      for (int kc = 0; kc < nchunk; ++kc, ++q) {
        const int s = q % NS;
        if (!f4_wait(&ready[s], (uint32_t)((q / NS) & 1), abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_try_wait(&full[s], (uint32_t)((q / NS) & 1));   // acquire: the copies the scale warps saw complete
          tc::fence_after_sync();
          const uint32_t st = smem_addr(stages + (size_t)s * kGuStage);
          const uint32_t sf = tmem + 256 + (uint32_t)(s * kGuSf);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_mxf4nvf4(tmem, tc::desc_sw128(st + 32 * kk), tc::desc_sw128(st + kGuA + 32 * kk), idesc,
                             sf + 4 * kk, sf + 16 + 8 * kk, (kc > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(&acc_full);
      __syncwarp();
    }
    if (lane == 0) {
      tc::mma_commit(&drain);
      mbar_wait_spin(&drain, 0u, kSpinLimit);
    }
  } else if (warp >= 6) {
    // ---- epilogue: warp w reads lanes 32 * (w % 4) .. + 31 and 16-value blocks 2 hh, 2 hh + 1
    const int qd = warp & 3, hh = (warp - 6) >> 2;
    const int rbi = p.I / 2 + p.I / 16;
    int ecur = 0, ntile = 0;
    F4Tile tl;
    for (int t = blockIdx.x; !*abort && f4_tile(t, ncb, rbpre, soff, E, ecur, tl); t += gridDim.x, ++ntile) {
      if (!f4_wait(&acc_full, (uint32_t)(ntile & 1), abort, true)) break;
      tc::fence_after_sync();
      const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
      const int m = 32 * qd + lane;
      const bool valid = m < tl.rows;
      const int row = tl.row0 + m;
      const float sg = __ldg(p.scales + 4 * tl.e + 0), su = __ldg(p.scales + 4 * tl.e + 1);
      uint32_t g16[2][16], u16[2][16];
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int blk = 2 * hh + j2;
        tc::tmem_ld16(tq + 16 * blk, g16[j2]);
        tc::tmem_ld16(tq + 128 + 16 * blk, u16[j2]);
      }
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&acc_empty);   // the accumulator is free for the next tile's MMAs
      uint32_t codes[4], sc = 0u;
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int blk = 2 * hh + j2;
        float a[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          a[j] = glu_act(__uint_as_float(g16[j2][j]) * sg, __uint_as_float(u16[j2][j]) * su, p.glu);
        uint32_t sbyte, c0, c1, hw[8];
        nvfp4_quant16(a, sbyte, c0, c1, hw);
        codes[2 * j2] = c0;
        codes[2 * j2 + 1] = c1;
        sc |= sbyte << (8 * j2);
        if (p.export_i16 && valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.i16 + (size_t)row * p.I + 128 * tl.cb + 16 * blk);
          dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        }
      }
      if (valid) {
        uint8_t* dst = p.in4 + (size_t)row * rbi;
        *reinterpret_cast<uint4*>(dst + 64 * tl.cb + 16 * hh) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        *reinterpret_cast<uint16_t*>(dst + p.I / 2 + 8 * tl.cb + 2 * hh) = (uint16_t)sc;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && abort_flag) atomicOr(p.err, kErrTimeout);
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

size_t pf4_gate_up_smem(int E) { return 1024 + (size_t)kGuStages * kGuStage + 8 * ((size_t)E + 1); }

// ------------------------------------------------------------------ launch

cudaError_t launch_prefill(const PfParams& p, cudaStream_t stream, const Pf4Params* fp4) {
  cudaError_t e;
  const int nsb = pf_sort_blocks(p.RT);
  const size_t sc = pf_count_smem(p.E), ss = pf_scatter_smem(p.E);
  if ((e = cudaFuncSetAttribute(k_pf_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(k_pf_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss)) != cudaSuccess)
    return e;
  k_pf_count<<<nsb, kSortThreads, sc, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_pf_scatter<<<nsb, kSortThreads, ss, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (fp4) {
    k_pf4_quant<<<(unsigned)((p.T + 7) / 8), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    const long long n = (long long)p.T * (p.mode == PF_W4A4 ? p.H / 16 : p.H / 32);
    k_pf_quant<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (fp4) return launch_prefill_fp4(*fp4, stream);
  const size_t sg = pf_gemm_smem();
  if (p.mode == PF_W4A8) {
    if ((e = cudaFuncSetAttribute(k_pf_gemm<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg)) !=
        cudaSuccess)
      return e;
    k_pf_gemm<0, true><<<sm_count(), kPfThreads, sg, stream>>>(p);
  } else {
    if ((e = cudaFuncSetAttribute(k_pf_gemm<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg)) !=
        cudaSuccess)
      return e;
    k_pf_gemm<0, false><<<sm_count(), kPfThreads, sg, stream>>>(p);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_pf_gemm<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg)) !=
      cudaSuccess)
    return e;
  k_pf_gemm<1, false><<<sm_count(), kPfThreads, sg, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const long long n = (long long)p.T * (p.H / 4);
    k_pf_combine<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_fp4(const Pf4Params& q, cudaStream_t stream) {
  cudaError_t e;
  const long long nsum = (long long)q.T * (q.H / 4);   // float4s of the fp32 token sums
  const size_t s0 = pf4_gate_up_smem(q.E), s1 = pf4_down_smem(q.E);
  if ((e = cudaFuncSetAttribute(k_pf4_gate_up, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s0)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_pf4_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)) != cudaSuccess)
    return e;
  k_pf4_gate_up<<<sm_count(), kGuThreads, s0, stream>>>(q);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_pf4_down<<<sm_count(), kF4Threads, s1, stream>>>(q);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (q.fixed) k_pf4_combine<<<(unsigned)((nsum + 255) / 256), 256, 0, stream>>>(q);
  else k_pf4_finish<<<(unsigned)((nsum + 255) / 256), 256, 0, stream>>>(q);
  return cudaGetLastError();
}

}  // namespace qre
