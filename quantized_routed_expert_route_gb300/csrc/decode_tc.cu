// Dense decode path for BF16 expert banks on the tensor cores.
//
// A BF16 bank row is a plain bf16 vector, so a decode pass over BF16 gate_up
// and down banks is, per selected expert, a small dense GEMM: the expert's
// rows times the hidden states of the tokens routed to it.  Raw BF16 expert
// rows go to a dense expert kernel instead of the quantized block-dot kernels
// (FreeToken issue #194, "perf(moe): avoid max-stride padding for
// heterogeneous GGUF expert banks", Proposed design), and a layer whose two
// projections are both BF16 takes the float path, with bf16 input and no
// requantized intermediate (FreeToken PR #704, "How it plugs into the CPU
// executor": the ("bf16", {}) spec, prep_input to bf16 / f32).  At batches
// the fused small-batch kernel cannot hold, four launches chained with
// programmatic dependent launch:
//
//   k_dt_route    every CTA sorts the routes by expert (stable) in shared
//                 memory; CTA 0 publishes the offsets and the permutation;
//                 all CTAs gather the bf16 x row of each sorted route into xs.
//   k_dt_gemm<0>  gate_up.  A tile is (expert, 128 intermediate columns,
//                 <= 128 routed tokens): per 64-wide K chunk a 2-D TMA brings
//                 the 128 gate rows, the 128 up rows (bf16, 128-byte swizzle)
//                 and the tokens' xs rows into one shared-memory stage; one
//                 thread issues tcgen05 kind::f16 MMAs (bf16 x bf16, fp32
//                 accumulation) into a gate and an up accumulator in tensor
//                 memory; four warps apply s_gate / s_up and SiLU-GLU in fp32
//                 and store the intermediate a, split as bf16 hi + lo.
//   k_dt_gemm<1>  down.  A tile is (expert, 128 output rows, <= 32 tokens); per K
//                 chunk the 128 down rows and the tokens' hi and lo rows; two
//                 MMAs per K step (hi, then lo, into one accumulator) carry a
//                 to ~2^-16; the epilogue scales by s_down * routing weight
//                 and stores fp32 per route.
//   k_dt_combine  out[t] = bf16(sum over k = 0..K-1 of the route rows), in
//                 route order, no atomics.
//
// Roles in a GEMM CTA (one CTA per SM, persistent over tiles): warp 0 lane 0
// issues the TMA loads into a ring of stages (4 for gate_up, 8 for down),
// warp 1 owns the tensor memory and its lane 0 issues the MMAs, warps 2..5
// run the epilogue from two alternating accumulator buffers.  Every wait is bounded in device time; on
// a timeout the CTA raises the error word, stops issuing, lets what it
// issued finish (bounded) and frees its tensor memory.
#include <cuda_bf16.h>

#include "decode_common.cuh"
#include "tc.cuh"

namespace qre {

namespace {

constexpr int kDtThreads = 192;                  // warp 0 TMA, warp 1 TMEM + MMA, warps 2..5 epilogue
constexpr int kDtRows = 128;                     // weight rows per tile (the MMA's M)
// Per-phase tile shape.  gate_up: <= 128 tokens (the MMA's N), 4 stages of
// 48 KB (16 KB gate + 16 KB up + <= 16 KB tokens).  down: a stage carries
// only 16 KB of weights (128 rows x 64 bf16), so tiles take <= 32 tokens and
// the ring has 8 stages of 24 KB (weights, then the hi and lo token rows):
// 128 KB of weights in flight per SM, enough to cover DRAM latency at this
// SM's share of the bandwidth.
template <int PHASE>
struct DtShape {
  static constexpr int kMaxN = PHASE == 0 ? 128 : 32;
  static constexpr int kStages = PHASE == 0 ? 4 : 8;
  static constexpr int kStageBytes = PHASE == 0 ? 48 * 1024 : 24 * 1024;
  static constexpr int kBOff = PHASE == 0 ? 32768 : 16384;     // token rows (down: the hi rows)
  static constexpr int kLoOff = 20480;                          // down: the lo rows
  static constexpr uint32_t kCols = PHASE == 0 ? 512 : 64;      // two accumulator buffers
};
constexpr int kDtMaxStages = 8;
constexpr int kDtEpiThreads = 128;
constexpr uint64_t kDtWaitNs = 2000000000ull;    // one wait gives up after 2 s of device time
constexpr int kRouteThreads = 512;

// 2-D tiled TMA load of the box at (x = column, y = row) of `map` into
// shared memory, completing its bytes on `bar`.
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

// Bounded wait on an mbarrier phase that also gives up once another role of
// the CTA has given up.  Returns false on timeout or abort.
__device__ __forceinline__ bool dt_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kDtWaitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ routes and gather

__global__ void __launch_bounds__(kRouteThreads) k_dt_route(const __grid_constant__ DtParams p) {
  extern __shared__ int rsm[];
  const int E = p.E, RT = p.RT;
  int* cnt = rsm;                                   // [16][E]
  int* base = cnt + (kRouteThreads / 32) * E;       // [E]
  int* wsum = base + E;                             // [33]
  int* off = wsum + 33;                             // [E+1]
  int* perm = off + E + 1;                          // [RT]
  pdl_wait();   // x and ids may come from the previous grid
  const bool bad = sort_routes_block(p.ids, RT, E, cnt, base, wsum, off, perm);
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int NV = off[E];
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kRouteThreads) p.off[e] = off[e];
    for (int s = tid; s < NV; s += kRouteThreads) p.perm[s] = perm[s];
    if (bad && (tid & 31) == 0) atomicOr(p.err, kErrBadId);
  }
  // xs[s] = x[token of sorted route s], 16 bytes per thread per step
  const int nq = p.H / 8;
  for (int s = blockIdx.x; s < NV; s += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)(perm[s] / p.K) * p.H);
    uint4* dst = reinterpret_cast<uint4*>(p.xs + (size_t)s * p.H);
    for (int q = tid; q < nq; q += kRouteThreads) dst[q] = __ldg(src + q);
  }
}

size_t dt_route_smem(int E, int RT) {
  return sizeof(int) * ((size_t)(kRouteThreads / 32) * E + E + 33 + (E + 1) + RT);
}

// ------------------------------------------------------------------ route sum

__global__ void k_dt_combine(const __grid_constant__ DtParams p) {
  pdl_wait();   // the down GEMM's y is complete
  pdl_launch_dependents();
  route_sum4(p.ids, p.y, p.out, p.T, p.K, p.E, p.H, (long long)blockIdx.x * blockDim.x + threadIdx.x);
}

// ------------------------------------------------------------------ grouped GEMMs

// Tile t of the persistent schedule: expert e (experts in order, tile_pre[e]
// = first tile of e), row block rb fastest, then token block.
struct DtTile {
  int e, rb, srow0, nv, n;   // expert, row block, first sorted row, valid tokens, MMA N (nv rounded up to 16)
};

template <int MAXN>
__device__ __forceinline__ DtTile dt_tile(const int* tile_pre, const int* offs, int E, int NB, int t) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_pre[mid] <= t) lo = mid;
    else hi = mid;
  }
  DtTile d;
  d.e = lo;
  const int tl = t - tile_pre[lo];
  d.rb = tl % NB;
  d.srow0 = offs[lo] + (tl / NB) * MAXN;
  d.nv = min(MAXN, offs[lo + 1] - d.srow0);
  d.n = (d.nv + 15) & ~15;
  return d;
}

// PHASE 0: gate_up (A = 128 gate rows and the 128 matching up rows, K = H;
// two accumulators per tile).  PHASE 1: down (A = 128 output rows, K = I; the
// hi and lo intermediate rows into one accumulator).
template <int PHASE>
__global__ void __launch_bounds__(kDtThreads, 1) k_dt_gemm(const __grid_constant__ DtParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Sh = DtShape<PHASE>;
  constexpr int kStages = Sh::kStages;
  __shared__ uint64_t full_bar[kDtMaxStages], empty_bar[kDtMaxStages], accf_bar[2], acce_bar[2], drain_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int tile_pre[kMaxE + 1];
  __shared__ int offs[kMaxE + 1];
  __shared__ int wsum[33];
  __shared__ volatile int abort_flag;
  constexpr uint32_t kCols = Sh::kCols;
  constexpr uint32_t kBufCols = kCols / 2;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const int NB = PHASE == 0 ? (p.I + kDtRows - 1) / kDtRows : (p.H + kDtRows - 1) / kDtRows;
  const int nK = (PHASE == 0 ? p.H : p.I) / 64;

  if (warp == 1) {
    tc::tmem_alloc(&tmem_base, kCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], kDtEpiThreads);
    }
    mbar_init(&drain_bar, 1);
    fence_mbar_init();
    prefetch_map(PHASE == 0 ? &p.map_gu : &p.map_dn);
    prefetch_map(PHASE == 0 ? &p.map_xs : &p.map_ih);
  }
  pdl_wait();   // PHASE 0: routes sorted and xs gathered; PHASE 1: the intermediate written
  for (int e = tid; e <= E; e += kDtThreads) offs[e] = __ldcg(p.off + e);
  __syncthreads();
  for (int e = tid; e < E; e += kDtThreads) {
    const int M = offs[e + 1] - offs[e];
    tile_pre[e] = ((M + Sh::kMaxN - 1) / Sh::kMaxN) * NB;
  }
  __syncthreads();
  const int total = block_exclusive_scan(tile_pre, E, wsum);
  pdl_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();   // weight rows: read once
      uint32_t g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const DtTile ti = dt_tile<Sh::kMaxN>(tile_pre, offs, E, NB, t);
        const int nb16 = ti.n >> 4;
        for (int kc = 0; kc < nK; ++kc, ++g) {
          const uint32_t s = g % kStages, u = g / kStages;
          if (u >= 1 && !dt_wait(&empty_bar[s], (u - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          uint8_t* st = base + s * Sh::kStageBytes;
          const int x = kc * 64;
          if (PHASE == 0) {
            mbar_arrive_expect_tx(&full_bar[s], 32768u + 2048u * (uint32_t)nb16);
            const int gy = ti.e * 2 * p.I + ti.rb * kDtRows;
            tma_load_2d_hint(st, &p.map_gu, x, gy, &full_bar[s], pol);
            tma_load_2d_hint(st + 16384, &p.map_gu, x, gy + p.I, &full_bar[s], pol);
            for (int j = 0; j < nb16; ++j)
              tma_load_2d(st + 32768 + 2048 * j, &p.map_xs, x, ti.srow0 + 16 * j, &full_bar[s]);
          } else {
            mbar_arrive_expect_tx(&full_bar[s], 16384u + 4096u * (uint32_t)nb16);
            tma_load_2d_hint(st, &p.map_dn, x, ti.e * p.H + ti.rb * kDtRows, &full_bar[s], pol);
            for (int j = 0; j < nb16; ++j) {
              tma_load_2d(st + Sh::kBOff + 2048 * j, &p.map_ih, x, ti.srow0 + 16 * j, &full_bar[s]);
              tma_load_2d(st + Sh::kLoOff + 2048 * j, &p.map_ih, x, p.RTp + ti.srow0 + 16 * j, &full_bar[s]);
            }
          }
        }
      }
      if (!ok) {
        atomicOr(p.err, kErrTimeout);
        // the copies already issued land before the CTA may exit (bounded)
        for (uint32_t j = (g > (uint32_t)kStages ? g - kStages : 0u); j < g; ++j)
          mbar_wait_spin(&full_bar[j % kStages], (j / kStages) & 1u, kDtWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      uint32_t g = 0, tcount = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tcount) {
        const DtTile ti = dt_tile<Sh::kMaxN>(tile_pre, offs, E, NB, t);
        const uint32_t bb = tcount & 1u, v = tcount >> 1;
        if (v >= 1 && !dt_wait(&acce_bar[bb], (v - 1) & 1u, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t idesc = tc::idesc_f16(kDtRows, (uint32_t)ti.n, true);
        const uint32_t d = tmem + bb * kBufCols;
        for (int kc = 0; kc < nK; ++kc, ++g) {
          const uint32_t s = g % kStages, u = g / kStages;
          if (!dt_wait(&full_bar[s], u & 1u, abort)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a0 = smem_addr(base + s * Sh::kStageBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
            if (PHASE == 0) {
              const uint64_t bd = tc::desc_sw128(a0 + 32768 + 32 * kk);
              tc::mma_f16(d, tc::desc_sw128(a0 + 32 * kk), bd, idesc, acc);
              tc::mma_f16(d + 128, tc::desc_sw128(a0 + 16384 + 32 * kk), bd, idesc, acc);
            } else {
              const uint64_t ad = tc::desc_sw128(a0 + 32 * kk);
              tc::mma_f16(d, ad, tc::desc_sw128(a0 + Sh::kBOff + 32 * kk), idesc, acc);
              tc::mma_f16(d, ad, tc::desc_sw128(a0 + Sh::kLoOff + 32 * kk), idesc, 1u);
            }
          }
          issued = true;
          tc::mma_commit(&empty_bar[s]);
        }
        if (!ok) break;
        tc::mma_commit(&accf_bar[bb]);
      }
      if (!ok) {
        atomicOr(p.err, kErrTimeout);
        if (issued) {   // the MMAs in flight finish before tensor memory is freed (bounded)
          tc::mma_commit(&drain_bar);
          mbar_wait_spin(&drain_bar, 0u, kDtWaitNs);
        }
      }
    }
  } else {
    // ---------------- epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31
    const int q = warp & 3;
    const int row = 32 * q + lane;
    uint32_t tcount = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
      const DtTile ti = dt_tile<Sh::kMaxN>(tile_pre, offs, E, NB, t);
      const uint32_t bb = tcount & 1u, v = tcount >> 1;
      if (!dt_wait(&accf_bar[bb], v & 1u, abort)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + bb * kBufCols;
      const int e = ti.e;
      if (PHASE == 0) {
        const int i = ti.rb * kDtRows + row;
        const bool vi = i < p.I;
        const float sg = __ldg(p.scales + 4 * e + 0), su = __ldg(p.scales + 4 * e + 1);
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          uint32_t g16[16], u16[16];
          tc::tmem_ld16(tq + c0, g16);
          tc::tmem_ld16(tq + 128 + c0, u16);
          tc::tmem_ld_wait();
          if (vi) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = c0 + j;
              if (c < ti.nv) {
                const int s = ti.srow0 + c;
                const float a = glu_act(__uint_as_float(g16[j]) * sg, __uint_as_float(u16[j]) * su, p.glu);
                const uint32_t hb = f32_to_bf16_bits_rn(a);
                const uint32_t lb = f32_to_bf16_bits_rn(a - __uint_as_float(hb << 16));
                p.ih[(size_t)s * p.I + i] = (uint16_t)hb;
                p.ih[(size_t)(p.RTp + s) * p.I + i] = (uint16_t)lb;
                p.inter[(size_t)__ldg(p.perm + s) * p.I + i] = a;
              }
            }
          }
        }
      } else {
        const int jr = ti.rb * kDtRows + row;
        const bool vj = jr < p.H;
        const float sd = __ldg(p.scales + 4 * e + 2);
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          uint32_t v16[16];
          tc::tmem_ld16(tq + c0, v16);
          tc::tmem_ld_wait();
          if (vj) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = c0 + j;
              if (c < ti.nv) {
                const int r = __ldg(p.perm + ti.srow0 + c);
                p.y[(size_t)r * p.H + jr] = __uint_as_float(v16[j]) * sd * __ldg(p.w + r);
              }
            }
          }
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&acce_bar[bb]);
    }
    if (!ok) atomicOr(p.err, kErrTimeout);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kCols);
}

template <int PHASE>
size_t dt_gemm_smem() { return 1024 + (size_t)DtShape<PHASE>::kStages * DtShape<PHASE>::kStageBytes; }

template <typename Kern>
cudaError_t launch_dt(Kern kernel, int grid, int threads, size_t smem, cudaStream_t stream, const DtParams& p) {
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

cudaError_t launch_dense(const DtParams& p, cudaStream_t stream) {
  const int G = sm_count();
  cudaError_t e;
  if ((e = launch_dt(k_dt_route, G, kRouteThreads, dt_route_smem(p.E, p.RT), stream, p)) != cudaSuccess) return e;
  if ((e = launch_dt(k_dt_gemm<0>, G, kDtThreads, dt_gemm_smem<0>(), stream, p)) != cudaSuccess) return e;
  if ((e = launch_dt(k_dt_gemm<1>, G, kDtThreads, dt_gemm_smem<1>(), stream, p)) != cudaSuccess) return e;
  const long long n = (long long)p.T * (p.H / 4);
  return launch_dt(k_dt_combine, (int)((n + 255) / 256), 256, 0, stream, p);
}

}  // namespace qre
