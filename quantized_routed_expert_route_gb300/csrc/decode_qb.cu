// Batched decode path for Q4_K banks.
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
// expert.  Five launches chained with programmatic dependent launch:
//
//   k_qb_route   every CTA sorts the routes by expert (stable) in shared
//                memory; CTA 0 publishes the offsets and the permutation; all
//                CTAs quantize the x row of each sorted route to q8_1 into
//                sorted planes (codes, 8-byte block records).
//   k_qb_gemm<0> gate_up.  A tile is (expert, 128 intermediate columns, <= 32
//                routed tokens).  Per 256-value K chunk one stage holds the
//                chunk's 144-byte super-block of the 128 gate rows and of the
//                128 up rows (2-D TMA, rows 144 bytes apart: conflict-free
//                16-byte loads) and the tokens' q8_1 codes and records.  A
//                thread owns a (gate, up) pair and half of each chunk's eight
//                blocks; it decodes each block once and accumulates its dot
//                products with every token (activation loads are
//                shared-memory broadcasts).  The two halves of a pair meet in
//                one shuffle; the epilogue applies s_gate / s_up and SiLU-GLU
//                in fp32 and stores the intermediate by route.
//   k_qb_requant prep_inter: the q8_1 of each sorted route's intermediate.
//   k_qb_gemm<1> down.  A tile is (expert, 256 output rows, <= 32 tokens), a
//                thread owns rows j and j+128; the epilogue scales by s_down *
//                routing weight and stores fp32 per route.
//   k_qb_combine out[t] = bf16(sum over k = 0..K-1 of the route rows), in
//                route order, no atomics.
//
// Every selected expert's rows are read from HBM once per pass (twice only
// for an expert with more than 32 routed tokens, the second time mostly from
// L2).  Every wait is bounded in device time; on a timeout the CTA raises the
// error word, stops issuing and lets its copies in flight land before exiting.
#include "decode_common.cuh"

namespace qre {

namespace {

constexpr int kQbConsumers = 256;                        // two weight rows x half the blocks per thread
constexpr int kQbThreads = kQbConsumers + 32;            // + one TMA producer warp (warp 8)
constexpr int kQbTok = 32;                               // routed tokens per tile
constexpr int kQbStages = 4;
constexpr int kQbSb = 144;                               // bytes of one Q4_K super-block (256 values) of a row
constexpr int kQbCodesOff = 256 * kQbSb;                 // 36,864: the 256 rows' super-blocks come first
constexpr int kQbRecOff = kQbCodesOff + kQbTok * 256;    // tokens' codes, 256 per token
constexpr int kQbStageBytes = kQbRecOff + kQbTok * 64;   // tokens' block records, 8 blocks x 8 bytes
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
  extern __shared__ int rsm[];
  const int E = p.E, RT = p.RT;
  int* cnt = rsm;                                    // [16][E]
  int* base = cnt + (kQbRouteThreads / 32) * E;      // [E]
  int* wsum = base + E;                              // [33]
  int* off = wsum + 33;                              // [E+1]
  int* perm = off + E + 1;                           // [RT]
  pdl_wait();   // x and ids may come from the previous grid
  const bool bad = sort_routes_block(p.ids, RT, E, cnt, base, wsum, off, perm);
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int NV = off[E];
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kQbRouteThreads) p.off[e] = off[e];
    for (int s = tid; s < NV; s += kQbRouteThreads) p.perm[s] = perm[s];
    if (bad && (tid & 31) == 0) atomicOr(p.err, kErrBadId);
  }
  const int nbh = p.H / 32;
  // sorted rows: the q8_1 of x[token of route perm[s]], one block per thread
  for (int s = blockIdx.x; s < NV; s += gridDim.x) {
    const uint16_t* xrow = p.x + (size_t)(perm[s] / p.K) * p.H;
    for (int b = tid; b < nbh; b += kQbRouteThreads) {
      uint32_t qw[8];
      float dh;
      int sum;
      uint16_t sh;
      quantize_x_block(xrow, b, qw, dh, sum, sh);
      uint4* qd = reinterpret_cast<uint4*>(p.aq + (size_t)s * p.H + 32 * b);
      qd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      qd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
      *reinterpret_cast<uint2*>(p.as + ((size_t)s * nbh + b) * 8) = make_uint2(__float_as_uint(dh), (uint32_t)sum);
    }
  }
  // the per-token planes the other decode paths leave in the workspace
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
      p.xd[t * nbh + b] = dh;
      p.xsum[t * nbh + b] = sum;
      p.xsh[t * nbh + b] = sh;
    }
  }
}

size_t qb_route_smem(int E, int RT) {
  return sizeof(int) * ((size_t)(kQbRouteThreads / 32) * E + E + 33 + (E + 1) + RT);
}

__global__ void k_qb_combine(const __grid_constant__ QbParams p) {
  pdl_wait();   // the down kernel's y is complete
  pdl_launch_dependents();
  route_sum4(p.ids, p.y, p.out, p.T, p.K, p.E, p.H, (long long)blockIdx.x * blockDim.x + threadIdx.x);
}

// q8_1 of the intermediate for the down kernel: sorted row s takes the fp32
// intermediate of route perm[s]; one 32-value block per thread.  The
// per-route planes the other paths leave are written too.
__global__ void k_qb_requant(const __grid_constant__ QbParams p) {
  pdl_wait();   // the gate_up kernel's intermediate is complete
  pdl_launch_dependents();
  const int nbi = p.I / 32;
  const int NV = __ldcg(p.off + p.E);
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= (long long)NV * nbi) return;
  const int s = (int)(b / nbi), blk = (int)(b - (long long)s * nbi);
  const int r = __ldcg(p.perm + s);
  float v[32];
  const float4* src = reinterpret_cast<const float4*>(p.inter + (size_t)r * p.I + 32 * blk);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = __ldcg(src + i);
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  uint32_t qw[8];
  float d;
  int sum;
  q8_1_quantize_block(v, qw, d, sum);
  const float dh = f16_bits_to_f32(f32_to_f16_bits_rn(d));
  uint4* qs = reinterpret_cast<uint4*>(p.iqs + (size_t)s * p.I + 32 * blk);
  qs[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  qs[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  *reinterpret_cast<uint2*>(p.iss + ((size_t)s * nbi + blk) * 8) = make_uint2(__float_as_uint(dh), (uint32_t)sum);
  uint4* qr = reinterpret_cast<uint4*>(p.iq + (size_t)r * p.I + 32 * blk);
  qr[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  qr[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  p.id[r * nbi + blk] = dh;
  p.isum[r * nbi + blk] = sum;
  p.ish[r * nbi + blk] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
}

// ------------------------------------------------------------------ grouped kernels

// Tile t of the persistent schedule: expert e (experts in order, tile_pre[e]
// = first tile of e), row block rb fastest, then token block.
struct QbTile {
  int e, rb, srow0, nv;   // expert, row block, first sorted row, tokens
};

__device__ __forceinline__ QbTile qb_tile(const int* tile_pre, const int* offs, int E, int NB, int t) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_pre[mid] <= t) lo = mid;
    else hi = mid;
  }
  QbTile d;
  d.e = lo;
  const int tl = t - tile_pre[lo];
  d.rb = tl % NB;
  d.srow0 = offs[lo] + (tl / NB) * kQbTok;
  d.nv = min(kQbTok, offs[lo + 1] - d.srow0);
  return d;
}

// Blocks 4h .. 4h+3 of one K chunk (a 256-value super-block) of the thread's
// two weight rows against the tile's tokens: each block decoded once, its
// integer dot with every token's q8_1 block scaled as d_a * (d*sc*dot -
// dmin*m*sum_a).
__device__ __forceinline__ void qb_chunk(const uint8_t* rowa, const uint8_t* rowb, const uint8_t* codes,
                                         const uint8_t* recs, int h, int nv, float (&acca)[kQbTok],
                                         float (&accb)[kQbTok]) {
#pragma unroll 1
  for (int j = 4 * h; j < 4 * h + 4; ++j) {
    int na[8], nb[8];
    float dsa, dma, dsb, dmb;
    q4k_decode(rowa, j, na, dsa, dma);
    q4k_decode(rowb, j, nb, dsb, dmb);
#pragma unroll
    for (int t = 0; t < kQbTok; ++t) {
      if (t >= nv) break;
      const uint8_t* c = codes + t * 256 + 32 * j;
      const uint4 c0 = lds128(c), c1 = lds128(c + 16);
      const uint2 rc = *reinterpret_cast<const uint2*>(recs + t * 64 + 8 * j);
      const int q[8] = {(int)c0.x, (int)c0.y, (int)c0.z, (int)c0.w, (int)c1.x, (int)c1.y, (int)c1.z, (int)c1.w};
      const float ad = __uint_as_float(rc.x), asum = (float)(int)rc.y;
      acca[t] += ad * (dsa * (float)int_dot8(na, q) - dma * asum);
      accb[t] += ad * (dsb * (float)int_dot8(nb, q) - dmb * asum);
    }
  }
}

// PHASE 0: gate_up (row a = gate row i, row b = up row I+i of a 128-pair
// tile, K = H).  PHASE 1: down (rows a, b = output rows j, j+128 of a
// 256-row tile, K = I).  Consumer thread (warp w, lane l): unit u = 16w +
// l%16 of the tile, blocks 4h..4h+3 of each chunk with h = l/16; the two
// halves of a unit are summed with one shuffle at the end of the tile.
template <int PHASE>
__global__ void __launch_bounds__(kQbThreads, 1) k_qb_gemm(const __grid_constant__ QbParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kQbStages], empty_bar[kQbStages];
  __shared__ int tile_pre[kMaxE + 1];
  __shared__ int offs[kMaxE + 1];
  __shared__ int wsum[33];
  __shared__ volatile int abort_flag;
  uint8_t* base = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
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
    fence_mbar_init();
    prefetch_map(PHASE == 0 ? &p.map_wgu : &p.map_wdn);
    prefetch_map(PHASE == 0 ? &p.map_aq : &p.map_iq);
    prefetch_map(PHASE == 0 ? &p.map_as : &p.map_is);
  }
  pdl_wait();   // PHASE 0: routes sorted and x quantized; PHASE 1: the intermediate requantized
  for (int e = tid; e <= E; e += kQbThreads) offs[e] = __ldcg(p.off + e);
  __syncthreads();
  for (int e = tid; e < E; e += kQbThreads) {
    const int M = offs[e + 1] - offs[e];
    tile_pre[e] = ((M + kQbTok - 1) / kQbTok) * NB;
  }
  __syncthreads();
  const int total = block_exclusive_scan(tile_pre, E, wsum);   // ends with a block barrier
  pdl_launch_dependents();
  volatile int* abort = &abort_flag;

  if (warp == kQbConsumers / 32) {
    // ---------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();   // weight rows: read once
      uint32_t g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const QbTile ti = qb_tile(tile_pre, offs, E, NB, t);
        for (int kc = 0; kc < nK; ++kc, ++g) {
          const uint32_t s = g % kQbStages, u = g / kQbStages;
          if (u >= 1 && !qb_wait(&empty_bar[s], (u - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          uint8_t* st = base + s * kQbStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], (uint32_t)kQbStageBytes);
          if (PHASE == 0) {
            const int y0 = ti.e * 2 * p.I + ti.rb * 128;
            tma_load_2d_hint(st, &p.map_wgu, kc * kQbSb, y0, &full_bar[s], pol);
            tma_load_2d_hint(st + 128 * kQbSb, &p.map_wgu, kc * kQbSb, y0 + p.I, &full_bar[s], pol);
            tma_load_2d(st + kQbCodesOff, &p.map_aq, kc * 256, ti.srow0, &full_bar[s]);
            tma_load_2d(st + kQbRecOff, &p.map_as, kc * 64, ti.srow0, &full_bar[s]);
          } else {
            const int y0 = ti.e * p.H + ti.rb * 256;
            tma_load_2d_hint(st, &p.map_wdn, kc * kQbSb, y0, &full_bar[s], pol);
            tma_load_2d_hint(st + 128 * kQbSb, &p.map_wdn, kc * kQbSb, y0 + 128, &full_bar[s], pol);
            tma_load_2d(st + kQbCodesOff, &p.map_iq, kc * 256, ti.srow0, &full_bar[s]);
            tma_load_2d(st + kQbRecOff, &p.map_is, kc * 64, ti.srow0, &full_bar[s]);
          }
        }
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

  // ---------------- consumers
  const int u = 16 * warp + (lane & 15), h = lane >> 4;
  uint32_t g = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
    const QbTile ti = qb_tile(tile_pre, offs, E, NB, t);
    float acca[kQbTok], accb[kQbTok];
#pragma unroll
    for (int i = 0; i < kQbTok; ++i) acca[i] = accb[i] = 0.f;
    for (int kc = 0; kc < nK; ++kc, ++g) {
      const uint32_t s = g % kQbStages, ph = (g / kQbStages) & 1u;
      if (!qb_wait(&full_bar[s], ph, abort)) {
        ok = false;
        break;
      }
      const uint8_t* st = base + s * kQbStageBytes;
      qb_chunk(st + u * kQbSb, st + (128 + u) * kQbSb, st + kQbCodesOff, st + kQbRecOff, h, ti.nv, acca, accb);
      mbar_arrive(&empty_bar[s]);
    }
    if (!ok) break;
#pragma unroll
    for (int i = 0; i < kQbTok; ++i) {
      if (i >= ti.nv) break;
      acca[i] += __shfl_xor_sync(0xffffffffu, acca[i], 16);
      accb[i] += __shfl_xor_sync(0xffffffffu, accb[i], 16);
    }
    const int e = ti.e;
    if (PHASE == 0) {
      // a = silu(h_gate * s_gate) * (h_up * s_up), by route; half h stores tokens of parity h
      const int i = ti.rb * 128 + u;
      const float sg = __ldg(p.scales + 4 * e + 0), su = __ldg(p.scales + 4 * e + 1);
#pragma unroll
      for (int k = 0; k < kQbTok; ++k) {
        if (k >= ti.nv) break;
        if ((k & 1) != h) continue;
        const int r = __ldcg(p.perm + ti.srow0 + k);
        p.inter[(size_t)r * p.I + i] = silu_glu(acca[k] * sg, accb[k] * su);
      }
    } else {
      const int j = ti.rb * 256 + u;
      const float sd = __ldg(p.scales + 4 * e + 2);
#pragma unroll
      for (int k = 0; k < kQbTok; ++k) {
        if (k >= ti.nv) break;
        if ((k & 1) != h) continue;
        const int r = __ldcg(p.perm + ti.srow0 + k);
        const float f = sd * __ldg(p.w + r);
        p.y[(size_t)r * p.H + j] = acca[k] * f;
        p.y[(size_t)r * p.H + j + 128] = accb[k] * f;
      }
    }
  }
  if (!ok) atomicOr(p.err, kErrTimeout);
}

size_t qb_gemm_smem() { return 128 + (size_t)kQbStages * kQbStageBytes; }

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
  if ((e = launch_qb(k_qb_route, G, kQbRouteThreads, qb_route_smem(p.E, p.RT), stream, p)) != cudaSuccess) return e;
  if ((e = launch_qb(k_qb_gemm<0>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
  {
    const long long n = (long long)p.RT * (p.I / 32);   // upper bound of the valid routes' blocks
    if ((e = launch_qb(k_qb_requant, (int)((n + 255) / 256), 256, 0, stream, p)) != cudaSuccess) return e;
  }
  if ((e = launch_qb(k_qb_gemm<1>, G, kQbThreads, qb_gemm_smem(), stream, p)) != cudaSuccess) return e;
  const long long n = (long long)p.T * (p.H / 4);
  return launch_qb(k_qb_combine, (int)((n + 255) / 256), 256, 0, stream, p);
}

}  // namespace qre
