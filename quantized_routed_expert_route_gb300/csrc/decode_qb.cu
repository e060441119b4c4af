// Batched decode path for Q4_K, Q4_0 and NVFP4 banks.
//
// At batches the fused small-batch kernel cannot hold, a Q4_K layer has
// several tokens routed to many of its selected experts.  The pass still
// computes, per route, the exact integer dot of each 32-value block of a
// weight row with the route's q8_1 activations, scaled by d * sc and
// corrected by dmin * m times the block's code sum (FreeToken PR #704, "How it
// plugs into the CPU executor": prep_input to q8_1, gate_up and down per row
// and route, prep_inter requantizing the intermediate; the Q4_K geometry of
// "perf(moe): avoid max-stride padding for heterogeneous GGUF expert banks",
// Reproduction geometry).  What changes is the order: each block of a
// weight row is decoded once and dotted with every routed token of its
// expert.  Four launches chained with programmatic dependent launch:
//
//   k_qb_route   quantizes every token's x to q8_1 once (codes and 8-byte
//                block records) and resets the tile counters.
//   k_qb_gemm<0> gate_up + prep_inter.  Every CTA first sorts the routes by
//                expert (stable) and orders the routed experts by route count
//                in shared memory, from the ids, before it waits on the route
//                kernel.  A tile is (expert, 128 intermediate columns, <= 8
//                routed tokens); tiles come from a global counter, heaviest
//                experts first.  Per 256-value K chunk one stage holds the
//                chunk's 144-byte super-block of the 128 gate rows and of the
//                128 up rows (2-D TMA, rows 144 bytes apart: conflict-free
//                16-byte loads) and each token's q8_1 codes and records (one
//                TMA row per token).  A thread owns a (gate, up) pair and a
//                quarter of each chunk's eight blocks: it decodes the chunk's
//                scales once, the 32-byte nibble run of its two blocks once,
//                and accumulates the block dots with every token (activation
//                loads are shared-memory broadcasts).  The quarters of a pair
//                meet in shared memory; the epilogue applies s_gate / s_up and
//                SiLU-GLU in fp32 and requantizes each warp's 32 intermediate
//                values to q8_1 (sorted rows for the down kernel, and by
//                route).
//   k_qb_gemm<1> down (the same prologue).  A tile is (expert, 256 output
//                rows, <= 8 tokens), a thread owns rows j and j+128; the
//                epilogue scales by s_down * routing weight and stores fp32
//                per route.
//   k_qb_combine out[t] = bf16(sum over k = 0..K-1 of the route rows), in
//                route order, no atomics.
//
// Every selected expert's rows are read from HBM once per pass (again, mostly
// from L2, for each further 8 routed tokens of an expert: small token blocks
// keep the tiles' costs even).  Every wait is bounded in device time; on a
// timeout the CTA raises the error word, stops issuing and lets its copies in
// flight land before exiting.
#include "decode_common.cuh"
#include "tc.cuh"

namespace qre {

namespace {

constexpr int kQbConsumers = 512;                        // two weight rows x a quarter of the blocks per thread
constexpr int kQbThreads = kQbConsumers + 32;            // + one TMA producer warp (warp 16)
constexpr int kQbTok = kQbTileTokens;                     // routed tokens per tile
constexpr int kQbStages = 4;
constexpr int kQbSb = 144;                               // bytes of one Q4_K super-block (256 values) of a row
// A stage: the 256 rows' super-blocks, then the tokens' codes (256 bytes a
// token), then their block records (8 blocks x 8 bytes a token).  Every
// tensor-copy destination is 128-byte aligned: gate_up copies each token's
// records on its own, so its record slots are 128 bytes apart; down copies
// the tile's tokens' records in one box, 64 bytes apart.
constexpr int kQbCodesOff = 256 * kQbSb;                 // 36,864
constexpr int kQbRecOff = kQbCodesOff + kQbTok * 256;    // 40,960
constexpr int kQbStageBytes = kQbRecOff + kQbTok * 128;  // 43,008
constexpr uint64_t kQbWaitNs = 2000000000ull;            // one wait gives up after 2 s of device time
constexpr int kQbRouteThreads = 512;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bounded wait that also gives up once another role of the CTA has.
__device__ __forceinline__ bool qb_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kQbWaitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// q8_1 of one 32-value block of a bf16 row; codes as eight int8x4 words, the
// fp16-rounded scale as fp32, the code sum, and fp16(d * sum).
__device__ __forceinline__ void quantize_x_block(const uint16_t* xrow, int b, uint32_t (&qw)[8], float& dh, int& sum,
                                                 uint16_t& sh) {
  float v[32];
  const uint4* src = reinterpret_cast<const uint4*>(xrow + 32 * b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[8 * i + j] = f[j];
  }
  float d;
  q8_1_quantize_block(v, qw, d, sum);
  dh = f16_bits_to_f32(f32_to_f16_bits_rn(d));
  sh = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
}

// ------------------------------------------------------------------ routes and activations

__global__ void __launch_bounds__(kQbRouteThreads) k_qb_route(const __grid_constant__ QbParams p) {
  pdl_wait();   // x and ids may come from the previous grid
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  if (blockIdx.x == 0 && tid == 0) {
    p.sched[0] = 0u;   // the tile counters of the two grouped kernels
    p.sched[1] = 0u;
  }
  // every token's q8_1, once: codes, records, and the planes left for inspection
  const int nbh = p.H / 32;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    const uint16_t* xrow = p.x + (size_t)t * p.H;
    for (int b = tid; b < nbh; b += kQbRouteThreads) {
      uint32_t qw[8];
      float dh;
      int sum;
      uint16_t sh;
      quantize_x_block(xrow, b, qw, dh, sum, sh);
      uint4* qd = reinterpret_cast<uint4*>(p.xq + (size_t)t * p.H + 32 * b);
      qd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      qd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
      *reinterpret_cast<uint2*>(p.xrec + ((size_t)t * nbh + b) * 8) = make_uint2(__float_as_uint(dh), (uint32_t)sum);
      p.xd[t * nbh + b] = dh;
      p.xsum[t * nbh + b] = sum;
      p.xsh[t * nbh + b] = sh;
    }
  }
}

__global__ void k_qb_combine(const __grid_constant__ QbParams p) {
  pdl_wait();   // the down kernel's y is complete
  pdl_launch_dependents();
  route_sum4(p.ids, p.y, p.out, p.T, p.K, p.E, p.H, (long long)blockIdx.x * blockDim.x + threadIdx.x);
}

// ------------------------------------------------------------------ grouped kernels

// What the producer tells the consumers about a stage: the tile's expert,
// row block, first sorted row, tokens (nv < 0: no more tiles) and the chunk.
struct __align__(16) QbMeta {
  int e, rb, srow0, nv_kc;   // nv_kc = nv | kc << 8
};

// d * sc and dmin * m of blocks 2q and 2q+1 of a Q4_K super-block, from its
// 16-byte header (d | dmin << 16, then the 12 packed 6-bit scale bytes).
__device__ __forceinline__ void q4k_scales2(const uint4 hdr, int q, float (&dsc)[2], float (&dmm)[2]) {
  const float d = f16_bits_to_f32(hdr.x & 0xFFFFu);
  const float dmin = f16_bits_to_f32(hdr.x >> 16);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = 2 * q + i;
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
    dsc[i] = d * (float)sc;
    dmm[i] = dmin * (float)m;
  }
}

// Blocks 2q and 2q+1 of one K chunk (a 256-value super-block) of the
// thread's two weight rows against the tile's tokens: the chunk's 32-byte
// nibble run q holds block 2q (low nibbles) and block 2q+1 (high nibbles);
// each block's integer dot with a token's q8_1 block is scaled as
// d_a * (d*sc*dot - dmin*m*sum_a).
template <int REC_PITCH>
__device__ __forceinline__ void qb_chunk(const uint8_t* rowa, const uint8_t* rowb, const uint8_t* codes,
                                         const uint8_t* recs, int q, int nv, float (&acca)[kQbTok],
                                         float (&accb)[kQbTok]) {
  float dsa[2], dma[2], dsb[2], dmb[2];
  q4k_scales2(lds128(rowa), q, dsa, dma);
  q4k_scales2(lds128(rowb), q, dsb, dmb);
  int al[8], ah[8], bl[8], bh[8];
  {
    const uint4 a0 = lds128(rowa + 16 + 32 * q), a1 = lds128(rowa + 32 + 32 * q);
    const uint4 b0 = lds128(rowb + 16 + 32 * q), b1 = lds128(rowb + 32 + 32 * q);
    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      al[i] = (int)(wa[i] & 0x0F0F0F0Fu);
      ah[i] = (int)((wa[i] >> 4) & 0x0F0F0F0Fu);
      bl[i] = (int)(wb[i] & 0x0F0F0F0Fu);
      bh[i] = (int)((wb[i] >> 4) & 0x0F0F0F0Fu);
    }
  }
#pragma unroll
  for (int t = 0; t < kQbTok; ++t) {
    if (t >= nv) break;
    const uint8_t* cp = codes + t * 256 + 64 * q;
    const uint4 q0 = lds128(cp), q1 = lds128(cp + 16), q2 = lds128(cp + 32), q3 = lds128(cp + 48);
    const uint4 rc = lds128(recs + t * REC_PITCH + 16 * q);   // (d, sum) of blocks 2q and 2q+1
    const int ql[8] = {(int)q0.x, (int)q0.y, (int)q0.z, (int)q0.w, (int)q1.x, (int)q1.y, (int)q1.z, (int)q1.w};
    const int qh[8] = {(int)q2.x, (int)q2.y, (int)q2.z, (int)q2.w, (int)q3.x, (int)q3.y, (int)q3.z, (int)q3.w};
    const float d0 = __uint_as_float(rc.x), s0 = (float)(int)rc.y;
    const float d1 = __uint_as_float(rc.z), s1 = (float)(int)rc.w;
    acca[t] += d0 * (dsa[0] * (float)int_dot8(al, ql) - dma[0] * s0);
    accb[t] += d0 * (dsb[0] * (float)int_dot8(bl, ql) - dmb[0] * s0);
    acca[t] += d1 * (dsa[1] * (float)int_dot8(ah, qh) - dma[1] * s1);
    accb[t] += d1 * (dsb[1] * (float)int_dot8(bh, qh) - dmb[1] * s1);
  }
}

// The 36 bytes of quarter Q (blocks 2Q and 2Q+1) of a row's Q4_0 K chunk
// (eight 18-byte blocks, 144 bytes, rows 144 bytes apart) as nine words:
// three conflict-free 16-byte loads from the 16-byte boundary 32Q at or below
// byte 36Q, of which words Q .. Q+8 are the quarter's (32Q + 48 >= 36Q + 36
// for Q <= 3, and 32Q + 48 <= 144).
template <int Q>
__device__ __forceinline__ void q4_0_quarter(const uint8_t* row, uint32_t (&w)[9]) {
  const uint4 a = lds128(row + 32 * Q), b = lds128(row + 32 * Q + 16), c = lds128(row + 32 * Q + 32);
  const uint32_t all[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 9; ++i) w[i] = all[Q + i];
}

// Unsigned codes (low nibbles: values 0..15, high: 16..31) and d of the two
// blocks of a quarter: block 2Q is bytes 0..17 (d, then codes from byte 2),
// block 2Q+1 bytes 18..35 (d in the high half of word 4, codes in words 5..8).
__device__ __forceinline__ void q4_0_quarter_codes(const uint32_t (&w)[9], int (&c0)[8], int (&c1)[8], float& d0,
                                                   float& d1) {
  d0 = f16_bits_to_f32(w[0] & 0xFFFFu);
  d1 = f16_bits_to_f32(w[4] >> 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = __funnelshift_r(w[i], w[i + 1], 16), y = w[5 + i];
    c0[i] = (int)(x & 0x0F0F0F0Fu);
    c0[i + 4] = (int)((x >> 4) & 0x0F0F0F0Fu);
    c1[i] = (int)(y & 0x0F0F0F0Fu);
    c1[i + 4] = (int)((y >> 4) & 0x0F0F0F0Fu);
  }
}

// Q4_0 blocks 2Q and 2Q+1 of one K chunk of rows a and b against the tile's
// tokens: each block's dot is d_a * d * (sum(q * a_q) - 8 * sum(a_q)).
template <int REC_PITCH, int Q>
__device__ __forceinline__ void qb_chunk_q4_0(const uint8_t* rowa, const uint8_t* rowb, const uint8_t* codes,
                                              const uint8_t* recs, int nv, float (&acca)[kQbTok],
                                              float (&accb)[kQbTok]) {
  int a0[8], a1[8], b0[8], b1[8];
  float da0, da1, db0, db1;
  {
    uint32_t w[9];
    q4_0_quarter<Q>(rowa, w);
    q4_0_quarter_codes(w, a0, a1, da0, da1);
    q4_0_quarter<Q>(rowb, w);
    q4_0_quarter_codes(w, b0, b1, db0, db1);
  }
#pragma unroll
  for (int t = 0; t < kQbTok; ++t) {
    if (t >= nv) break;
    const uint8_t* cp = codes + t * 256 + 64 * Q;
    const uint4 q0 = lds128(cp), q1 = lds128(cp + 16), q2 = lds128(cp + 32), q3 = lds128(cp + 48);
    const uint4 rc = lds128(recs + t * REC_PITCH + 16 * Q);   // (d, sum) of blocks 2Q and 2Q+1
    const int ql[8] = {(int)q0.x, (int)q0.y, (int)q0.z, (int)q0.w, (int)q1.x, (int)q1.y, (int)q1.z, (int)q1.w};
    const int qh[8] = {(int)q2.x, (int)q2.y, (int)q2.z, (int)q2.w, (int)q3.x, (int)q3.y, (int)q3.z, (int)q3.w};
    const float e0 = __uint_as_float(rc.x), e1 = __uint_as_float(rc.z);
    const int s0 = 8 * (int)rc.y, s1 = 8 * (int)rc.w;
    acca[t] += e0 * (da0 * (float)(int_dot8(a0, ql) - s0));
    accb[t] += e0 * (db0 * (float)(int_dot8(b0, ql) - s0));
    acca[t] += e1 * (da1 * (float)(int_dot8(a1, qh) - s1));
    accb[t] += e1 * (db1 * (float)(int_dot8(b1, qh) - s1));
  }
}

// NVFP4 blocks 2q and 2q+1 of one K chunk for rows a and b (unit u of the
// tile): each row's 128 code bytes sit in a 128-byte-swizzled tile (16-byte
// chunk j of row u at position j ^ (u % 8)), its 16 UE4M3 bytes at scl + 16u
// (word q holds the four scales of blocks 2q and 2q+1).  Each 32-value
// block's two 16-value integer dots with a token's q8_1 block are scaled as
// d_a * 0.5 * (scale_0 * dot_0 + scale_1 * dot_1).
template <int REC_PITCH>
__device__ __forceinline__ void qb_chunk_nvfp4(const uint8_t* ca, const uint8_t* cb, const uint8_t* sla,
                                               const uint8_t* slb, int u, const uint8_t* codes, const uint8_t* recs,
                                               int q, int nv, float (&acca)[kQbTok], float (&accb)[kQbTok]) {
  const uint32_t swa = lds32(sla + 16 * u + 4 * q), swb = lds32(slb + 16 * u + 4 * q);
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = 2 * q + jj;
    // sign-split words (two dp4a per word and token): most tiles of a
    // decode batch hold one or two tokens, where this beats converting the
    // words to signed bytes first (measured on the T=8 layer)
    uint32_t pa[8], na[8], pb[8], nb[8];
    nvfp4_words(lds128(ca + tc::sw128_chunk(u, j)), pa, na);
    nvfp4_words(lds128(cb + tc::sw128_chunk(u, j)), pb, nb);
    const float2 fa = ue4m3x2_to_float2((uint16_t)(swa >> (16 * jj)));
    const float2 fb = ue4m3x2_to_float2((uint16_t)(swb >> (16 * jj)));
#pragma unroll
    for (int t = 0; t < kQbTok; ++t) {
      if (t >= nv) break;
      const uint8_t* cp = codes + t * 256 + 32 * j;
      const uint4 q0 = lds128(cp), q1 = lds128(cp + 16);
      const int qv[8] = {(int)q0.x, (int)q0.y, (int)q0.z, (int)q0.w, (int)q1.x, (int)q1.y, (int)q1.z, (int)q1.w};
      const float ad = *reinterpret_cast<const float*>(recs + t * REC_PITCH + 8 * j);
      int a0, a1, b0, b1;
      nvfp4_int_dots(pa, na, qv, a0, a1);
      nvfp4_int_dots(pb, nb, qv, b0, b1);
      acca[t] += ad * 0.5f * (fa.x * (float)a0 + fa.y * (float)a1);
      accb[t] += ad * 0.5f * (fb.x * (float)b0 + fb.y * (float)b1);
    }
  }
}

// PHASE 0: gate_up (row a = gate row i, row b = up row I+i of a 128-pair
// tile, K = H).  PHASE 1: down (rows a, b = output rows j, j+128 of a
// 256-row tile, K = I).  Consumer warp w takes blocks 2q and 2q+1 of each
// chunk (q = w/4, a quarter of the chunk) for the 32 units 32*(w%4) .. +31 of
// the tile, one per lane, so a warp's activation loads are broadcasts and a
// warp of quarter 0 holds 32 consecutive intermediate values (one q8_1
// block).  At the end of a tile quarters 1..3 hand their partial sums to
// quarter 0 through shared memory (two mbarriers, bounded waits), which adds
// them in quarter order and runs the epilogue.
template <int PHASE, int WT>
__global__ void __launch_bounds__(kQbThreads, 1) k_qb_gemm(const __grid_constant__ QbParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kQbStages], empty_bar[kQbStages], xfull_bar, xfree_bar;
  __shared__ QbMeta smeta[kQbStages];
  __shared__ int tile_pre[kMaxE + 1];
  __shared__ int offs[kMaxE + 1];
  __shared__ int eord[kMaxE];
  __shared__ int perm_s[kMaxTopK * kTChunk];   // route index of each sorted row
  __shared__ int wsum[33];
  __shared__ volatile int abort_flag;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);   // swizzled tiles need 1024
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const int NB = PHASE == 0 ? p.I / 128 : p.H / 256;
  const int nK = (PHASE == 0 ? p.H : p.I) / 256;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kQbStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kQbConsumers);
    }
    mbar_init(&xfull_bar, kQbConsumers - 128);   // quarters 1..3
    mbar_init(&xfree_bar, 128);                  // quarter 0
    fence_mbar_init();
    prefetch_map(PHASE == 0 ? &p.map_wgu : &p.map_wdn);
    if (WT == W_NVFP4) prefetch_map(PHASE == 0 ? &p.map_wgus : &p.map_wdns);
    prefetch_map(PHASE == 0 ? &p.map_xq : &p.map_iq);
    prefetch_map(PHASE == 0 ? &p.map_xr : &p.map_is);
  }
  // The routes sorted by expert (stable) and the routed experts ordered by
  // route count (most first, then by id), computed by every CTA from the ids
  // before waiting on the previous grid: the ids were complete before the
  // route kernel let this grid launch (it waits first, then lets dependents
  // launch).  The scratch lives in the stage ring, which no copy has touched.
  int U, total;
  {
    const int RT = p.RT;
    int* cnt = reinterpret_cast<int*>(base);        // [warps][E]
    int* bse = cnt + (kQbThreads / 32) * E;          // [E]
    int* cm = bse + E;                               // [RT+1]: experts per route count, then positions
    const bool bad = sort_routes_block(p.ids, RT, E, cnt, bse, wsum, offs, perm_s);
    if (PHASE == 0 && blockIdx.x == 0 && bad && lane == 0) atomicOr(p.err, kErrBadId);
    for (int i = tid; i <= RT; i += kQbThreads) cm[i] = 0;
    __syncthreads();
    for (int e = tid; e < E; e += kQbThreads) {
      const int M = offs[e + 1] - offs[e];
      if (M > 0) atomicAdd(&cm[RT - M], 1);
    }
    __syncthreads();
    U = block_exclusive_scan(cm, RT + 1, wsum);
    if (warp == 0) {
      // experts in id order, each placed after the earlier ones of its count
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int M = (e < E) ? offs[e + 1] - offs[e] : 0;
        const bool v = M > 0;
        const unsigned peers = __match_any_sync(0xffffffffu, v ? M : -1 - lane);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (v) eord[cm[RT - M] + rank] = e;
        __syncwarp();
        if (v && rank == 0) cm[RT - M] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    for (int i = tid; i < U; i += kQbThreads) {
      const int e = eord[i];
      tile_pre[i] = ((offs[e + 1] - offs[e] + kQbTok - 1) / kQbTok) * NB;
    }
    __syncthreads();
    total = block_exclusive_scan(tile_pre, U, wsum);   // ends with a block barrier
  }
  pdl_wait();   // PHASE 0: x quantized, counters reset; PHASE 1: the intermediate requantized
  pdl_launch_dependents();
  volatile int* abort = &abort_flag;

  if (warp == kQbConsumers / 32) {
    // ---------------- TMA producer: tiles from the global counter, most routes first
    if (lane == 0) {
      fence_proxy_async_smem();   // the prologue's scratch writes come before the copies into the ring
      const uint64_t pol = l2_policy_evict_first();   // weight rows: read once
      uint32_t g = 0;
      bool ok = true;
      int tok[kQbTok];
      for (;;) {
        const int t = (int)atomicAdd(p.sched + PHASE, 1u);
        const uint32_t s0 = g % kQbStages, u0 = g / kQbStages;
        if (t >= total) {
          // no tile left: a stage with nv < 0 tells the consumers to stop
          if (u0 >= 1 && !qb_wait(&empty_bar[s0], (u0 - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          smeta[s0] = QbMeta{0, 0, 0, -1};
          mbar_arrive(&full_bar[s0]);
          break;
        }
        int lo = 0, hi = U;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (tile_pre[mid] <= t) lo = mid;
          else hi = mid;
        }
        const int e = eord[lo];
        const int tl = t - tile_pre[lo];
        const int rb = tl % NB;
        const int srow0 = offs[e] + (tl / NB) * kQbTok;
        const int nv = min(kQbTok, offs[e + 1] - srow0);
        if (PHASE == 0)
          for (int i = 0; i < nv; ++i) tok[i] = perm_s[srow0 + i] / p.K;
        for (int kc = 0; kc < nK; ++kc, ++g) {
          const uint32_t s = g % kQbStages, u = g / kQbStages;
          if (u >= 1 && !qb_wait(&empty_bar[s], (u - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          smeta[s] = QbMeta{e, rb, srow0, nv | (kc << 8)};
          uint8_t* st = base + s * kQbStageBytes;
          // rows a (box at ya) and b (box at yb) of the tile: 36,864 bytes in both formats
          const int ya = PHASE == 0 ? e * 2 * p.I + rb * 128 : e * p.H + rb * 256;
          const int yb = PHASE == 0 ? ya + p.I : ya + 128;
          const CUtensorMap* mw = PHASE == 0 ? &p.map_wgu : &p.map_wdn;
          mbar_arrive_expect_tx(&full_bar[s], PHASE == 0 ? (uint32_t)(kQbCodesOff + nv * 320)
                                                         : (uint32_t)(kQbRecOff + kQbTok * 64));
          if (WT == W_Q4_K || WT == W_Q4_0) {   // both 144 bytes per 256-value chunk of a row
            tma_load_2d_hint(st, mw, kc * kQbSb, ya, &full_bar[s], pol);
            tma_load_2d_hint(st + 128 * kQbSb, mw, kc * kQbSb, yb, &full_bar[s], pol);
          } else {
            const CUtensorMap* ms = PHASE == 0 ? &p.map_wgus : &p.map_wdns;
            const int xs = (PHASE == 0 ? p.H : p.I) / 2 + kc * 16;
            tma_load_2d_hint(st, mw, kc * 128, ya, &full_bar[s], pol);
            tma_load_2d_hint(st + 16384, mw, kc * 128, yb, &full_bar[s], pol);
            tma_load_2d_hint(st + 32768, ms, xs, ya, &full_bar[s], pol);
            tma_load_2d_hint(st + 34816, ms, xs, yb, &full_bar[s], pol);
          }
          if (PHASE == 0) {
            for (int i = 0; i < nv; ++i) {
              tma_load_2d(st + kQbCodesOff + 256 * i, &p.map_xq, kc * 256, tok[i], &full_bar[s]);
              tma_load_2d(st + kQbRecOff + 128 * i, &p.map_xr, kc * 64, tok[i], &full_bar[s]);
            }
          } else {
            tma_load_2d(st + kQbCodesOff, &p.map_iq, kc * 256, srow0, &full_bar[s]);
            tma_load_2d(st + kQbRecOff, &p.map_is, kc * 64, srow0, &full_bar[s]);
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        atomicOr(p.err, kErrTimeout);
        // the copies already issued land before the CTA may exit (bounded)
        for (uint32_t j = (g > (uint32_t)kQbStages ? g - kQbStages : 0u); j < g; ++j)
          mbar_wait_spin(&full_bar[j % kQbStages], (j / kQbStages) & 1u, kQbWaitNs);
      }
    }
    return;
  }

  // ---------------- consumers: follow the producer's stages
  const int u = 32 * (warp & 3) + lane, q = warp >> 2;
  float2* xch = reinterpret_cast<float2*>(base + (size_t)kQbStages * kQbStageBytes);   // [3][kQbTok][128]
  float acca[kQbTok], accb[kQbTok];
  bool ok = true;
  uint32_t ntile = 0;
  for (uint32_t g = 0;; ++g) {
    const uint32_t s = g % kQbStages, ph = (g / kQbStages) & 1u;
    if (!qb_wait(&full_bar[s], ph, abort)) {
      ok = false;
      break;
    }
    const QbMeta m = smeta[s];
    if (m.nv_kc < 0) break;
    const int nv = m.nv_kc & 0xFF, kc = m.nv_kc >> 8;
    if (kc == 0) {
#pragma unroll
      for (int i = 0; i < kQbTok; ++i) acca[i] = accb[i] = 0.f;
    }
    const uint8_t* st = base + s * kQbStageBytes;
    if (WT == W_Q4_K) {
      qb_chunk<PHASE == 0 ? 128 : 64>(st + u * kQbSb, st + (128 + u) * kQbSb, st + kQbCodesOff, st + kQbRecOff, q,
                                      nv, acca, accb);
    } else if (WT == W_Q4_0) {
      constexpr int RP = PHASE == 0 ? 128 : 64;
      const uint8_t *ra = st + u * kQbSb, *rb = st + (128 + u) * kQbSb;
      switch (q) {   // warp-uniform: the quarter's word offset is a compile-time constant
        case 0: qb_chunk_q4_0<RP, 0>(ra, rb, st + kQbCodesOff, st + kQbRecOff, nv, acca, accb); break;
        case 1: qb_chunk_q4_0<RP, 1>(ra, rb, st + kQbCodesOff, st + kQbRecOff, nv, acca, accb); break;
        case 2: qb_chunk_q4_0<RP, 2>(ra, rb, st + kQbCodesOff, st + kQbRecOff, nv, acca, accb); break;
        default: qb_chunk_q4_0<RP, 3>(ra, rb, st + kQbCodesOff, st + kQbRecOff, nv, acca, accb); break;
      }
    } else
      qb_chunk_nvfp4<PHASE == 0 ? 128 : 64>(st, st + 16384, st + 32768, st + 34816, u, st + kQbCodesOff,
                                            st + kQbRecOff, q, nv, acca, accb);
    mbar_arrive(&empty_bar[s]);
    if (kc != nK - 1) continue;
    // ---- the tile is complete: quarters 1..3 hand over, quarter 0 finishes
    const uint32_t n = ntile++;
    if (q != 0) {
      if (n >= 1 && !qb_wait(&xfree_bar, (n - 1) & 1u, abort)) {
        ok = false;
        break;
      }
      float2* xq = xch + (q - 1) * kQbTok * 128;
#pragma unroll
      for (int k = 0; k < kQbTok; ++k) {
        if (k >= nv) break;
        xq[k * 128 + u] = make_float2(acca[k], accb[k]);
      }
      mbar_arrive(&xfull_bar);
      continue;
    }
    if (!qb_wait(&xfull_bar, n & 1u, abort)) {
      ok = false;
      break;
    }
#pragma unroll
    for (int k = 0; k < kQbTok; ++k) {
      if (k >= nv) break;
#pragma unroll
      for (int qq = 0; qq < 3; ++qq) {
        const float2 o = xch[(qq * kQbTok + k) * 128 + u];
        acca[k] += o.x;
        accb[k] += o.y;
      }
    }
    mbar_arrive(&xfree_bar);
    const int e = m.e;
    if (PHASE == 0) {
      // prep_inter: a = silu(h_gate * s_gate) * (h_up * s_up) in fp32, then
      // the q8_1 of the warp's 32 values for every token, sorted and by route
      const int i = m.rb * 128 + u;
      const int nbi = p.I / 32, blk = i / 32;
      const float sg = __ldg(p.scales + 4 * e + 0), su = __ldg(p.scales + 4 * e + 1);
#pragma unroll
      for (int k = 0; k < kQbTok; ++k) {
        if (k >= nv) break;
        const int srow = m.srow0 + k;
        const int r = perm_s[srow];
        const float a = glu_act(acca[k] * sg, accb[k] * su, p.glu);
        float d;
        int sum;
        const int q = q8_1_quantize_lane(a, d, sum);
        const float dh = f16_bits_to_f32(f32_to_f16_bits_rn(d));
        p.inter[(size_t)r * p.I + i] = a;
        p.iqs[(size_t)srow * p.I + i] = (int8_t)q;
        p.iq[(size_t)r * p.I + i] = (int8_t)q;
        if (lane == 0) {
          *reinterpret_cast<uint2*>(p.iss + ((size_t)srow * nbi + blk) * 8) =
              make_uint2(__float_as_uint(dh), (uint32_t)sum);
          p.id[r * nbi + blk] = dh;
          p.isum[r * nbi + blk] = sum;
          p.ish[r * nbi + blk] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
        }
      }
    } else {
      const int j = m.rb * 256 + u;
      const float sd = __ldg(p.scales + 4 * e + 2);
#pragma unroll
      for (int k = 0; k < kQbTok; ++k) {
        if (k >= nv) break;
        const int r = perm_s[m.srow0 + k];
        const float f = sd * __ldg(p.w + r);
        p.y[(size_t)r * p.H + j] = acca[k] * f;
        p.y[(size_t)r * p.H + j + 128] = accb[k] * f;
      }
    }
  }
  if (!ok) atomicOr(p.err, kErrTimeout);
}

size_t qb_gemm_smem() { return 1024 + (size_t)kQbStages * kQbStageBytes + 3 * (size_t)kQbTok * 128 * sizeof(float2); }

template <typename Kern>
cudaError_t launch_qb(Kern kernel, int grid, int threads, size_t smem, cudaStream_t stream, const QbParams& p) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

cudaError_t launch_qbatch(const QbParams& p, cudaStream_t stream) {
  const int G = sm_count();
  cudaError_t e;
  if ((e = launch_qb(k_qb_route, G, kQbRouteThreads, 0, stream, p)) != cudaSuccess) return e;
  if (p.wt == W_NVFP4) {
    if ((e = launch_qb(k_qb_gemm<0, W_NVFP4>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
    if ((e = launch_qb(k_qb_gemm<1, W_NVFP4>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
  } else if (p.wt == W_Q4_0) {
    if ((e = launch_qb(k_qb_gemm<0, W_Q4_0>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
    if ((e = launch_qb(k_qb_gemm<1, W_Q4_0>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
  } else {
    if ((e = launch_qb(k_qb_gemm<0, W_Q4_K>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
    if ((e = launch_qb(k_qb_gemm<1, W_Q4_K>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
  }
  const long long n = (long long)p.T * (p.H / 4);
  return launch_qb(k_qb_combine, (int)((n + 255) / 256), 256, 0, stream, p);
}

}  // namespace qre
