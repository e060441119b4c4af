// Device code shared by the decode kernels (decode.cu) and the fused
// small-batch layer kernel (layer_small.cu): route grouping, TMA stage
// issue, activation staging, q8_1 quantization into shared memory and the
// per-block dot loops.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace qre {

constexpr int kThreads = 256;                 // k_prep and the test hooks
constexpr int kConsumerWarps = 8;             // decode kernels: 8 consumer warps ...
constexpr int kProducerWarp = kConsumerWarps; // ... and one TMA producer warp
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 1);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int NT = 4;                         // routes per work item held in registers
constexpr uint32_t kWaitLimit = 8192;         // sleeping polls of a barrier (~4 s) before giving up
constexpr uint32_t kErrBadId = 1u, kErrTimeout = 2u;

// Named barrier 1 synchronises the NTH consumer threads only (the producer
// warp may already have left).
template <int NTH = kConsumerThreads>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTH) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ------------------------------------------------------------------ grouping

struct GroupSmem {
  int* slot_of;     // [E]   expert -> slot (valid for experts that are routed to)
  int* slot_e;      // [S]   slot -> expert, ascending expert id
  int* slot_off;    // [S+1] start of each slot's routes in `routes`
  int* cursor;      // [S]
  int* misc;        // [8]   0: slot count, 1: bad id seen, 2..5: pair range, 6: abort, 7: stages issued
  int* wsum;        // [33]
  float* sscale;    // [3*S] s_gate, s_up, s_down of each slot's expert
  int16_t* routes;  // [T*K] route indices t*K+k grouped by slot, route order inside a slot
  int16_t* rtok;    // [T*K] token t of each entry of `routes`
};

__host__ __device__ inline size_t group_smem_bytes(int E, int RT) {
  const int S = E < RT ? E : RT;
  return sizeof(int) * (size_t)(E + S + (S + 1) + S + 8 + 33 + 3 * S) + 2 * sizeof(int16_t) * (size_t)RT + 16;
}

__device__ inline GroupSmem carve_group(uint8_t* base, int E, int RT) {
  const int S = E < RT ? E : RT;
  GroupSmem g;
  int* p = reinterpret_cast<int*>(base);
  g.slot_of = p; p += E;
  g.slot_e = p; p += S;
  g.slot_off = p; p += S + 1;
  g.cursor = p; p += S;
  g.misc = p; p += 8;
  g.wsum = p; p += 33;
  g.sscale = reinterpret_cast<float*>(p); p += 3 * S;
  g.routes = reinterpret_cast<int16_t*>(p);
  g.rtok = g.routes + RT;
  return g;
}

// Exclusive prefix sum of a[0..n) in place (whole block); returns the total.
__device__ inline int block_exclusive_scan(int* a, int n, int* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nw = nthr >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int local = 0;
  for (int i = b0; i < b1; ++i) local += a[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = (lane < nw) ? wsum[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < nw) wsum[lane] = inc - v;
    if (lane == nw - 1) wsum[32] = inc;
  }
  __syncthreads();
  int run = wsum[warp] + incl - local;
  for (int i = b0; i < b1; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  const int total = wsum[32];
  __syncthreads();
  return total;
}

// Stable sort of routes 0..RT-1 by expert id, by the whole block: per-warp
// expert counts over contiguous route ranges, an exclusive scan over experts,
// then each warp places its routes (match/rank inside each group of 32), so
// the rows of an expert keep route order.  Routes whose id is outside [0, E)
// are left out.  Scratch in shared memory: cnt [warps][E], base [E], wsum
// [33].  Results: off[e] = first sorted row of expert e, off[E] = valid
// routes, perm[row] = route index (shared or global memory), complete for the
// whole block on return.  Returns, in every lane of a warp, whether that warp
// saw an invalid id.
__device__ inline bool sort_routes_block(const int32_t* ids, int RT, int E, int* cnt, int* base, int* wsum, int* off,
                                         int* perm) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nthr = blockDim.x, NW = nthr >> 5;
  for (int i = tid; i < NW * E; i += nthr) cnt[i] = 0;
  __syncthreads();
  const int per = (RT + NW - 1) / NW;
  const int r0 = min(RT, w * per), r1 = min(RT, r0 + per);
  bool bad = false;
  for (int r = r0 + lane; r < r1; r += 32) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&cnt[w * E + e], 1);
    else bad = true;
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    int acc = 0;
    for (int ww = 0; ww < NW; ++ww) {
      const int c = cnt[ww * E + e];
      cnt[ww * E + e] = acc;
      acc += c;
    }
    base[e] = acc;
  }
  __syncthreads();
  const int total = block_exclusive_scan(base, E, wsum);
  for (int e = tid; e < E; e += nthr) off[e] = base[e];
  if (tid == 0) off[E] = total;
  for (int rb = r0; rb < r1; rb += 32) {
    const int r = rb + lane;
    const int e = (r < r1) ? ids[r] : -1;
    const bool v = r < r1 && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (v) perm[base[e] + cnt[w * E + e] + rank] = r;
    __syncwarp();
    if (v && rank == 0) cnt[w * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  return __any_sync(0xffffffffu, bad);
}

// Route sum of the grouped paths, four outputs per thread: for element
// idx of [T][H/4], out[t][n..n+3] = bf16(sum over k = 0..K-1, in route order,
// of y[t*K+k][n..n+3]) over the routes whose expert id is valid; one
// rounding to bf16, no atomics.
__device__ __forceinline__ void route_sum4(const int32_t* ids, const float* y, uint16_t* out, int T, int K, int E,
                                           int H, long long idx) {
  const int nq = H / 4;
  if (idx >= (long long)T * nq) return;
  const int t = (int)(idx / nq), n = 4 * (int)(idx - (long long)t * nq);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < K; ++k) {
    const int r = t * K + k;
    const int e = __ldg(ids + r);
    if (e < 0 || e >= E) continue;
    const float4 v = __ldcg(reinterpret_cast<const float4*>(y + (size_t)r * H + n));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  uint2 o;
  o.x = f32_to_bf16_bits_rn(acc.x) | (f32_to_bf16_bits_rn(acc.y) << 16);
  o.y = f32_to_bf16_bits_rn(acc.z) | (f32_to_bf16_bits_rn(acc.w) << 16);
  *reinterpret_cast<uint2*>(out + (size_t)t * H + n) = o;
}

constexpr int kGroupWarpRoutes = 128;   // routes one warp groups (four per lane)

// Group up to kGroupWarpRoutes routes with one warp: an expert histogram in
// slot_of, a warp scan over the experts in ascending order gives each routed
// expert its slot and the start of its routes, then match/rank places every
// route after the earlier routes of the same expert.
__device__ inline void group_routes_warp(const int32_t* ids, int RT, int E, int K, const GroupSmem& g, int lane) {
  for (int e = lane; e < E; e += 32) g.slot_of[e] = 0;
  __syncwarp();
  int ev[4];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int r = 32 * c + lane;
    ev[c] = (r < RT) ? ids[r] : -1;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int r = 32 * c + lane;
    const bool v = r < RT && ev[c] >= 0 && ev[c] < E;
    bad |= (r < RT && !v);
    if (v) atomicAdd(&g.slot_of[ev[c]], 1);
  }
  __syncwarp();
  const int per = (E + 31) >> 5, e0 = lane * per;
  int cnt = 0, pres = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      const int h = g.slot_of[e];
      cnt += h;
      pres += (h > 0) ? 1 : 0;
    }
  }
  int ci = cnt, pi = pres;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, ci, o), y = __shfl_up_sync(0xffffffffu, pi, o);
    if (lane >= o) {
      ci += x;
      pi += y;
    }
  }
  const int S = __shfl_sync(0xffffffffu, pi, 31), NV = __shfl_sync(0xffffffffu, ci, 31);
  int co = ci - cnt, po = pi - pres;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      const int h = g.slot_of[e];
      if (h > 0) {
        g.slot_of[e] = po;
        g.slot_e[po] = e;
        g.slot_off[po] = co;
        g.cursor[po] = co;
        ++po;
        co += h;
      }
    }
  }
  if (lane == 0) {
    g.slot_off[S] = NV;
    g.misc[0] = S;
  }
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (32 * c >= RT) break;
    const int r = 32 * c + lane;
    const bool v = r < RT && ev[c] >= 0 && ev[c] < E;
    const unsigned peers = __match_any_sync(0xffffffffu, v ? ev[c] : -1 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (v) {
      const int pos = g.cursor[g.slot_of[ev[c]]] + rank;
      g.routes[pos] = (int16_t)r;
      g.rtok[pos] = (int16_t)(r / K);
    }
    __syncwarp();
    if (v && rank == 0) g.cursor[g.slot_of[ev[c]]] += __popc(peers);
    __syncwarp();
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) g.misc[1] = bad ? 1 : 0;
}

// Group up to 32 routes with one warp (lane r holds route r): match/shuffle
// give each distinct valid expert its slot (ascending id) and each route its
// place after the earlier routes of the same expert.
__device__ inline void group_routes_small_warp(const int32_t* ids, int RT, int E, int K, const GroupSmem& g,
                                               int lane) {
  int e = (lane < RT) ? ids[lane] : -1;
  const bool valid = (lane < RT) && e >= 0 && e < E;
  const bool bad = (lane < RT) && !valid;
  const int key = valid ? e : -1 - lane;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const bool first = valid && (lane == __ffs(peers) - 1);
  int slot = 0, off = 0;
  for (int j = 0; j < RT; ++j) {   // lanes >= RT hold no route
    const int ej = __shfl_sync(0xffffffffu, key, j);
    const int fj = __shfl_sync(0xffffffffu, first ? 1 : 0, j);
    const unsigned pj = __shfl_sync(0xffffffffu, peers, j);
    if (valid && fj && ej < key) {
      ++slot;
      off += __popc(pj);
    }
  }
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid) {
    g.routes[off + rank] = (int16_t)lane;
    g.rtok[off + rank] = (int16_t)(lane / K);
  }
  if (first) {
    g.slot_e[slot] = e;
    g.slot_off[slot] = off;
  }
  const unsigned firsts = __ballot_sync(0xffffffffu, first);
  const unsigned valids = __ballot_sync(0xffffffffu, valid);
  const unsigned bads = __ballot_sync(0xffffffffu, bad);
  if (lane == 0) {
    g.slot_off[__popc(firsts)] = __popc(valids);
    g.misc[0] = __popc(firsts);
    g.misc[1] = bads ? 1 : 0;
  }
}

// Group the T*K routes by expert: the distinct valid experts in ascending id
// order become slots; each slot lists its routes in route order.  Reads only
// `ids`.  Every CTA of a kernel computes the same grouping.  Up to 32 routes
// one warp does it with match/shuffle, up to 128 one warp with a histogram;
// beyond that the whole block scans.
__device__ inline void group_routes(const int32_t* ids, int RT, int E, int K, const GroupSmem& g) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x;
  if (RT <= 32) {
    if (warp == 0) group_routes_small_warp(ids, RT, E, K, g, lane);
    __syncthreads();
    return;
  }
  if (RT <= kGroupWarpRoutes) {
    if (warp == 0) group_routes_warp(ids, RT, E, K, g, lane);
    __syncthreads();
    return;
  }
  for (int e = tid; e < E; e += nthr) g.slot_of[e] = 0;
  if (tid == 0) g.misc[1] = 0;
  __syncthreads();
  for (int r = tid; r < RT; r += nthr) {
    const int e = ids[r];
    if (e >= 0 && e < E) g.slot_of[e] = 1;
    else g.misc[1] = 1;
  }
  __syncthreads();
  const int S = block_exclusive_scan(g.slot_of, E, g.wsum);
  for (int e = tid; e < E; e += nthr) {
    const int nxt = (e + 1 < E) ? g.slot_of[e + 1] : S;
    if (nxt != g.slot_of[e]) g.slot_e[g.slot_of[e]] = e;
  }
  for (int s = tid; s < S; s += nthr) g.cursor[s] = 0;
  __syncthreads();
  for (int r = tid; r < RT; r += nthr) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&g.cursor[g.slot_of[e]], 1);
  }
  __syncthreads();
  for (int s = tid; s < S; s += nthr) g.slot_off[s] = g.cursor[s];
  __syncthreads();
  const int tot = block_exclusive_scan(g.slot_off, S, g.wsum);
  if (tid == 0) g.slot_off[S] = tot;
  for (int s = tid; s < S; s += nthr) g.cursor[s] = g.slot_off[s];
  __syncthreads();
  if (warp == 0) {
    for (int base = 0; base < RT; base += 32) {
      const int r = base + lane;
      int s = -1;
      if (r < RT) {
        const int e = ids[r];
        if (e >= 0 && e < E) s = g.slot_of[e];
      }
      const unsigned peers = __match_any_sync(0xffffffffu, s);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (s >= 0) {
        g.routes[g.cursor[s] + rank] = (int16_t)r;
        g.rtok[g.cursor[s] + rank] = (int16_t)(r / K);
      }
      __syncwarp();
      if (s >= 0 && rank == 0) g.cursor[s] += __popc(peers);
      __syncwarp();
    }
  }
  if (tid == 0) g.misc[0] = S;
  __syncthreads();
}

// ------------------------------------------------------------------ activations

template <bool kBf16In>
__device__ __forceinline__ void load_block32(const void* src, int b, float (&v)[32]) {
  if constexpr (kBf16In) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + (size_t)b * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[8];
      bf16x8_to_f32(__ldg(p + i), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * i + j] = f[j];
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + (size_t)b * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = __ldcg(p + i);
      v[4 * i + 0] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
    }
  }
}


// ------------------------------------------------------------------ gate_up

struct PairCursor {
  int u, i;
};

// Next stage of at most `ps` pairs, staying inside one slot and before (ue, ie).
__device__ __forceinline__ bool next_gu_stage(PairCursor& c, int ue, int ie, int I, int ps, int& su, int& si,
                                              int& sn) {
  if (c.u > ue || (c.u == ue && c.i >= ie)) return false;
  const int lim = (c.u == ue) ? ie : I;
  su = c.u;
  si = c.i;
  sn = min(ps, lim - c.i);
  c.i += sn;
  if (c.i >= I) {
    c.u += 1;
    c.i = 0;
  }
  return true;
}

// First pair (u, i) whose cumulative cost start is >= target; (S, 0) if none.
// The remainder inside one slot is below cost * I < 2^32, so the division is
// 32-bit.
__device__ inline void pair_at_cost(long long target, const int* slot_off, int S, int I, int w0, int& u, int& i) {
  long long c = 0;
  for (u = 0; u < S; ++u) {
    const unsigned cs = (unsigned)(w0 + (slot_off[u + 1] - slot_off[u]));
    const long long span = (long long)cs * I;
    if (c + span > target) {
      const long long rem = target - c;
      i = rem <= 0 ? 0 : (int)(((unsigned)rem + cs - 1u) / cs);
      if (i >= I) {
        u += 1;
        i = 0;
      }
      return;
    }
    c += span;
  }
  u = S;
  i = 0;
}

// pair_at_cost computed by one warp (all 32 lanes call it with the same
// arguments; the result is valid in every lane): slot costs 1 + routes, in
// chunks of 32 slots with a warp scan instead of a serial walk.
__device__ inline void pair_at_cost_warp(long long target, const int* slot_off, int S, int I, int w0, int lane,
                                         int& u, int& i) {
  long long run = 0;
  for (int base = 0; base < S; base += 32) {
    const int sl = base + lane;
    const int c = (sl < S) ? w0 + (slot_off[sl + 1] - slot_off[sl]) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const long long start = (run + (incl - c)) * I, end = (run + incl) * I;
    const unsigned hit = __ballot_sync(0xffffffffu, sl < S && start <= target && target < end);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const long long st = __shfl_sync(0xffffffffu, start, l);
      const int cs = __shfl_sync(0xffffffffu, c, l);
      const long long rem = target - st;
      u = base + l;
      i = rem <= 0 ? 0 : (int)(((unsigned)rem + (unsigned)cs - 1u) / (unsigned)cs);
      if (i >= I) {
        u += 1;
        i = 0;
      }
      return;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  u = S;
  i = 0;
}

// floor(W * c / G) for the CTA boundaries, through fp64 (exact below 2^53).
__device__ __forceinline__ long long cost_cut(long long W, int c, int G) {
  return (long long)floor((double)W * (double)c / (double)G);
}

__device__ __forceinline__ const uint8_t* align16_down(const uint8_t* a) {
  return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15));
}
__device__ __forceinline__ uint32_t round16(uint32_t v) { return (v + 15u) & ~15u; }

__device__ inline void issue_gu_stage(const DecodeParams& p, uint8_t* buf, uint64_t* bar, int e, int i0, int n,
                               uint64_t pol) {
  const size_t rb = (size_t)p.rb_gu;
  const uint8_t* gsrc = p.gu_bank + ((size_t)e * 2 * p.I + i0) * rb;
  const uint8_t* usrc = p.gu_bank + ((size_t)e * 2 * p.I + p.I + i0) * rb;
  const uint8_t* ga = align16_down(gsrc);
  const uint8_t* ua = align16_down(usrc);
  const uint32_t gsz = round16((uint32_t)(gsrc - ga) + (uint32_t)(n * rb));
  const uint32_t usz = round16((uint32_t)(usrc - ua) + (uint32_t)(n * rb));
  mbar_arrive_expect_tx(bar, gsz + usz);
  tma_load_1d(buf, ga, gsz, bar, pol);
  tma_load_1d(buf + p.gu_up_off, ua, usz, bar, pol);
}

// Copy `bytes` (a multiple of 4; both pointers 16-byte aligned when bytes is a
// multiple of 16) from global memory (written by an earlier grid) into shared
// memory with the consumer warps, four independent 16-byte loads per thread
// per round.
template <int NTH = kConsumerThreads>
__device__ inline void copy_to_smem(void* dst, const void* src, size_t bytes) {
  const int tid = threadIdx.x;
  if ((bytes & 15) == 0) {
    const size_t n = bytes / 16;
    const int4* s = static_cast<const int4*>(src);
    int4* d = static_cast<int4*>(dst);
    for (size_t i = tid; i < n; i += 4 * NTH) {
      int4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * NTH < n) v[j] = __ldcg(s + i + j * NTH);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * NTH < n) d[i + j * NTH] = v[j];
    }
  } else {
    const size_t n = bytes / 4;
    const int* s = static_cast<const int*>(src);
    int* d = static_cast<int*>(dst);
    for (size_t i = tid; i < n; i += NTH) d[i] = __ldcg(s + i);
  }
}

// Where a kernel reads its q8_1 (or float) activations from: shared memory
// when they were staged there, else the workspace.  Row r of the codes is at
// q + r*n, its block scales at d + r*(n/32), code sums at s + r*(n/32); float
// activations (BF16 rows) are bf16 x (xb) or the fp32 intermediate (xf).
struct ActSrc {
  const int8_t* q;
  const float* d;
  const int* s;
  const uint16_t* xb;
  const float* xf;
  int n;
};

__device__ __forceinline__ ActQ8 act_block(const ActSrc& a, int row, int blk) {
  ActQ8 r;
  const int4* p = reinterpret_cast<const int4*>(a.q + (size_t)row * a.n + 32 * blk);
  const int4 lo = p[0], hi = p[1];
  r.q[0] = lo.x; r.q[1] = lo.y; r.q[2] = lo.z; r.q[3] = lo.w;
  r.q[4] = hi.x; r.q[5] = hi.y; r.q[6] = hi.z; r.q[7] = hi.w;
  const size_t bi = (size_t)row * (a.n / 32) + blk;
  r.d = a.d[bi];
  r.sum = a.s[bi];
  return r;
}

// Accumulate one 32-value block b of a quantized row into acc[0..nt).
template <int WT, int NTT>
__device__ __forceinline__ void accum_q_block(const uint8_t* row, int k, int b, const ActQ8 (&a)[NTT], int nt,
                                              float (&acc)[NTT]) {
  if constexpr (WT == W_NVFP4 || WT == W_NVFP4_U) {
    uint32_t pos[8], neg[8];
    float2 s;
    nvfp4_decode<WT == W_NVFP4>(row, k, b, pos, neg, s);
    if constexpr (NTT >= 3) {
      int w[8];
      nvfp4_signed(pos, neg, w);
#pragma unroll
      for (int t = 0; t < NTT; ++t) {
        if (t < nt) {
          int d0, d1;
          int_dots_halves(w, a[t].q, d0, d1);
          acc[t] += a[t].d * 0.5f * (s.x * (float)d0 + s.y * (float)d1);
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < NTT; ++t) {
        if (NTT == 1 || t < nt) {
          int d0, d1;
          nvfp4_int_dots(pos, neg, a[t].q, d0, d1);
          acc[t] += a[t].d * 0.5f * (s.x * (float)d0 + s.y * (float)d1);
        }
      }
    }
  } else if constexpr (WT == W_Q4_K) {
    int nib[8];
    float dsc, dmm;
    q4k_decode(row, b, nib, dsc, dmm);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) {
        const int dd = int_dot8(nib, a[t].q);
        acc[t] += a[t].d * (dsc * (float)dd - dmm * (float)a[t].sum);
      }
    }
  } else if constexpr (WT == W_Q6_K) {
    int wq[8];
    float d, s0, s1;
    q6k_decode(row, b, wq, d, s0, s1);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) {
        int d0, d1;
        int_dots_halves(wq, a[t].q, d0, d1);
        acc[t] += (d * a[t].d) * (s0 * (float)d0 + s1 * (float)d1);
      }
    }
  } else if constexpr (WT == W_Q4_0) {
    int wq[8];
    float d;
    q4_0_decode(row, b, wq, d);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += (d * a[t].d) * (float)(int_dot8(wq, a[t].q) - 8 * a[t].sum);
    }
  } else if constexpr (WT == W_Q4_1 || WT == W_Q5_1) {
    int wq[8];
    float d, m;
    if constexpr (WT == W_Q4_1) q4_1_decode(row, b, wq, d, m);
    else q5_1_decode(row, b, wq, d, m);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += a[t].d * (d * (float)int_dot8(wq, a[t].q) + m * (float)a[t].sum);
    }
  } else if constexpr (WT == W_Q5_0) {
    int wq[8];
    float d;
    q5_0_decode(row, b, wq, d);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += (d * a[t].d) * (float)(int_dot8(wq, a[t].q) - 16 * a[t].sum);
    }
  } else if constexpr (WT == W_Q5_K) {
    int wq[8];
    float dsc, dmm;
    q5k_decode(row, b, wq, dsc, dmm);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += a[t].d * (dsc * (float)int_dot8(wq, a[t].q) - dmm * (float)a[t].sum);
    }
  } else if constexpr (WT == W_MXFP4) {
    int wq[8];
    float sc;
    mxfp4_decode(row, b, wq, sc);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += (a[t].d * sc * 0.5f) * (float)int_dot8(wq, a[t].q);
    }
  } else {  // W_Q8_0
    static_assert(WT == W_Q8_0 || is_float_w(WT), "unhandled weight type");  // float rows: unreachable instantiations
    int wq[8];
    float d;
    q8_0_decode(row, b, wq, d);
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) acc[t] += (d * a[t].d) * (float)int_dot8(wq, a[t].q);
    }
  }
}

// One gate_up work item: the gate row and the up row of one pair against up
// to NTT routes' activations, over blocks [b0, b1) striped across the lanes.
// Results are warp-reduced and valid in every lane.
template <int WT, int NTT>
__device__ __forceinline__ void gu_item(const uint8_t* grow, const uint8_t* urow, int H, int b0, int b1, int lane,
                                        const ActSrc& act, const int (&tok)[NT], int nt, float (&ag)[NT],
                                        float (&au)[NT]) {
  float accg[NTT], accu[NTT];
#pragma unroll
  for (int t = 0; t < NTT; ++t) accg[t] = accu[t] = 0.f;
  if constexpr (is_float_w(WT)) {
    for (int c = b0 + lane; c < b1; c += 32) {
      float wg[8], wu[8];
      float_row_chunk8<WT>(grow, c, wg);
      float_row_chunk8<WT>(urow, c, wu);
#pragma unroll
      for (int t = 0; t < NTT; ++t) {
        if (NTT == 1 || t < nt) {
          float xv[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(act.xb + (size_t)tok[t] * H + 8 * c), xv);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            accg[t] = fmaf(wg[j], xv[j], accg[t]);
            accu[t] = fmaf(wu[j], xv[j], accu[t]);
          }
        }
      }
    }
  } else {
    int b = b0 + lane;
    // two blocks per lane per iteration (four independent decode/dot chains)
    // when few routes share the item; several routes already give that ILP
    for (; NTT <= 2 && b + 32 < b1; b += 64) {
      ActQ8 a0[NTT], a1[NTT];
#pragma unroll
      for (int t = 0; t < NTT; ++t)
        if (NTT == 1 || t < nt) {
          a0[t] = act_block(act, tok[t], b);
          a1[t] = act_block(act, tok[t], b + 32);
        }
      accum_q_block<WT, NTT>(grow, H, b, a0, nt, accg);
      accum_q_block<WT, NTT>(urow, H, b, a0, nt, accu);
      accum_q_block<WT, NTT>(grow, H, b + 32, a1, nt, accg);
      accum_q_block<WT, NTT>(urow, H, b + 32, a1, nt, accu);
    }
    for (; b < b1; b += 32) {
      ActQ8 a[NTT];
#pragma unroll
      for (int t = 0; t < NTT; ++t)
        if (NTT == 1 || t < nt) a[t] = act_block(act, tok[t], b);
      accum_q_block<WT, NTT>(grow, H, b, a, nt, accg);
      accum_q_block<WT, NTT>(urow, H, b, a, nt, accu);
    }
  }
#pragma unroll
  for (int t = 0; t < NTT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      accg[t] += __shfl_xor_sync(0xffffffffu, accg[t], o);
      accu[t] += __shfl_xor_sync(0xffffffffu, accu[t], o);
    }
    ag[t] = accg[t];
    au[t] = accu[t];
  }
}

// silu(g) * u in fp32: expf (about 1 ulp) and a 2-ulp division.
// One (gate, up) pair against one activation row held in shared memory as
// q8_1 planes (codes aq[H], scales ad[H/32], code sums as[H/32]): blocks
// striped across the 32 lanes, two per lane per iteration; returns the
// warp-reduced (h_gate, h_up) in every lane.
template <int WT>
__device__ __forceinline__ float2 gu_pair_q8(const uint8_t* grow, const uint8_t* urow, int H, int lane,
                                             const int8_t* aq, const float* ad, const int* as) {
  const int nb = H >> 5;
  float accg[1] = {0.f}, accu[1] = {0.f};
  int b = lane;
  for (; b + 32 < nb; b += 64) {
    ActQ8 a0[1], a1[1];
    {
      const int4* p0 = reinterpret_cast<const int4*>(aq + 32 * b);
      const int4* p1 = reinterpret_cast<const int4*>(aq + 32 * (b + 32));
      const int4 l0 = p0[0], h0 = p0[1], l1 = p1[0], h1 = p1[1];
      a0[0].q[0] = l0.x; a0[0].q[1] = l0.y; a0[0].q[2] = l0.z; a0[0].q[3] = l0.w;
      a0[0].q[4] = h0.x; a0[0].q[5] = h0.y; a0[0].q[6] = h0.z; a0[0].q[7] = h0.w;
      a1[0].q[0] = l1.x; a1[0].q[1] = l1.y; a1[0].q[2] = l1.z; a1[0].q[3] = l1.w;
      a1[0].q[4] = h1.x; a1[0].q[5] = h1.y; a1[0].q[6] = h1.z; a1[0].q[7] = h1.w;
      a0[0].d = ad[b]; a0[0].sum = as[b];
      a1[0].d = ad[b + 32]; a1[0].sum = as[b + 32];
    }
    accum_q_block<WT, 1>(grow, H, b, a0, 1, accg);
    accum_q_block<WT, 1>(urow, H, b, a0, 1, accu);
    accum_q_block<WT, 1>(grow, H, b + 32, a1, 1, accg);
    accum_q_block<WT, 1>(urow, H, b + 32, a1, 1, accu);
  }
  for (; b < nb; b += 32) {
    ActQ8 a[1];
    const int4* p0 = reinterpret_cast<const int4*>(aq + 32 * b);
    const int4 l0 = p0[0], h0 = p0[1];
    a[0].q[0] = l0.x; a[0].q[1] = l0.y; a[0].q[2] = l0.z; a[0].q[3] = l0.w;
    a[0].q[4] = h0.x; a[0].q[5] = h0.y; a[0].q[6] = h0.z; a[0].q[7] = h0.w;
    a[0].d = ad[b]; a[0].sum = as[b];
    accum_q_block<WT, 1>(grow, H, b, a, 1, accg);
    accum_q_block<WT, 1>(urow, H, b, a, 1, accu);
  }
  float g = accg[0], u = accu[0];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    g += __shfl_xor_sync(0xffffffffu, g, o);
    u += __shfl_xor_sync(0xffffffffu, u, o);
  }
  return make_float2(g, u);
}

// One row per LPR-lane group against one route's intermediate held in shared
// memory as q8_1 planes; reduced within the lane group.
template <int WT, int LPR>
__device__ __forceinline__ float dn_row_q8(const uint8_t* rowp, bool vrow, int I, int sl, const int8_t* aq,
                                           const float* ad, const int* as) {
  const int nbi = I >> 5;
  float acc[1] = {0.f};
  if (vrow) {
    int b = sl;
    for (; b + LPR < nbi; b += 2 * LPR) {
      ActQ8 a0[1], a1[1];
      const int4* p0 = reinterpret_cast<const int4*>(aq + 32 * b);
      const int4* p1 = reinterpret_cast<const int4*>(aq + 32 * (b + LPR));
      const int4 l0 = p0[0], h0 = p0[1], l1 = p1[0], h1 = p1[1];
      a0[0].q[0] = l0.x; a0[0].q[1] = l0.y; a0[0].q[2] = l0.z; a0[0].q[3] = l0.w;
      a0[0].q[4] = h0.x; a0[0].q[5] = h0.y; a0[0].q[6] = h0.z; a0[0].q[7] = h0.w;
      a1[0].q[0] = l1.x; a1[0].q[1] = l1.y; a1[0].q[2] = l1.z; a1[0].q[3] = l1.w;
      a1[0].q[4] = h1.x; a1[0].q[5] = h1.y; a1[0].q[6] = h1.z; a1[0].q[7] = h1.w;
      a0[0].d = ad[b]; a0[0].sum = as[b];
      a1[0].d = ad[b + LPR]; a1[0].sum = as[b + LPR];
      accum_q_block<WT, 1>(rowp, I, b, a0, 1, acc);
      accum_q_block<WT, 1>(rowp, I, b + LPR, a1, 1, acc);
    }
    for (; b < nbi; b += LPR) {
      ActQ8 a[1];
      const int4* p0 = reinterpret_cast<const int4*>(aq + 32 * b);
      const int4 l0 = p0[0], h0 = p0[1];
      a[0].q[0] = l0.x; a[0].q[1] = l0.y; a[0].q[2] = l0.z; a[0].q[3] = l0.w;
      a[0].q[4] = h0.x; a[0].q[5] = h0.y; a[0].q[6] = h0.z; a[0].q[7] = h0.w;
      a[0].d = ad[b]; a[0].sum = as[b];
      accum_q_block<WT, 1>(rowp, I, b, a, 1, acc);
    }
  }
  float v = acc[0];
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The GLU of the layer: act(g) * u, act = SiLU (kind 0) or the tanh form of
// GELU (kind 1): silu(g) = g / (1 + exp(-g)); gelu_tanh(g) =
// g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3))) (Hendrycks and Gimpel,
// "Gaussian Error Linear Units", 2016).  FreeToken PR #732, "Other checks",
// runs its experts with both.
constexpr int kGluSilu = 0, kGluGeluTanh = 1;
// gelu_tanh(g) * u, out of line: it keeps tanhf's code out of every kernel's
// hot path when the layer uses SiLU
static __device__ __noinline__ float gelu_tanh_glu(float g, float u) {
  const float z = 0.7978845608028654f * fmaf(0.044715f * g, g * g, g);
  return 0.5f * g * (1.0f + tanhf(z)) * u;
}
__device__ __forceinline__ float glu_act(float g, float u, int kind) {
  if (kind == kGluGeluTanh) return gelu_tanh_glu(g, u);
  return __fdividef(g, 1.0f + expf(-g)) * u;
}

// Quantize `nblk` 32-value blocks (row-major values from `src`) into q8_1
// planes in shared memory -- codes q[32*b + i], scales d[b] (fp16 values as
// fp32), code sums sm[b] -- one block per consumer thread.  When `ids` is
// given, blocks of routes (rows of `blocks_per_row` blocks) with an invalid
// expert id are skipped.  With `mirror`, the blocks also go to the workspace
// planes (wq, wd, wsum, wsh) for inspection.
template <bool kBf16In, int NTH = kConsumerThreads>
__device__ inline void quantize_blocks_to_smem(const void* src, int nblk, const int32_t* ids, int E, int blocks_per_row,
                                        int8_t* q, float* d, int* sm, bool mirror, int8_t* wq, float* wd, int* wsum,
                                        uint16_t* wsh) {
  for (int b = threadIdx.x; b < nblk; b += NTH) {
    if (ids) {
      const int e = ids[b / blocks_per_row];
      if (e < 0 || e >= E) continue;
    }
    float v[32];
    load_block32<kBf16In>(src, b, v);
    uint32_t qw[8];
    float dd;
    int sum;
    q8_1_quantize_block(v, qw, dd, sum);
    const float dh = f16_bits_to_f32(f32_to_f16_bits_rn(dd));
    uint4* qd = reinterpret_cast<uint4*>(q + (size_t)b * 32);
    qd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    qd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    d[b] = dh;
    sm[b] = sum;
    if (mirror) {
      uint4* wqd = reinterpret_cast<uint4*>(wq + (size_t)b * 32);
      wqd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      wqd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
      wd[b] = dh;
      wsum[b] = sum;
      wsh[b] = (uint16_t)f32_to_f16_bits_rn(dd * (float)sum);
    }
  }
}

// ------------------------------------------------------------------ down

struct DownStage {
  int js, nr, u0, ns;
};

__device__ __forceinline__ DownStage down_stage(int k, int S, int nj, int rs, int sps) {
  const int ngrp = (S + sps - 1) / sps;
  DownStage d;
  d.js = (k / ngrp) * rs;
  d.nr = min(rs, nj - d.js);
  d.u0 = (k % ngrp) * sps;
  d.ns = min(sps, S - d.u0);
  return d;
}

__device__ inline void issue_dn_stage(const DecodeParams& p, uint8_t* buf, uint64_t* bar, const GroupSmem& g,
                               const DownStage& st, int j0, uint64_t pol) {
  uint32_t total = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int i = 0; i < st.ns; ++i) {
      const int e = g.slot_e[st.u0 + i];
      const uint8_t* s = p.dn_bank + ((size_t)e * p.H + j0 + st.js) * p.rb_dn;
      const uint8_t* a = align16_down(s);
      const uint32_t sz = round16((uint32_t)(s - a) + (uint32_t)(st.nr * p.rb_dn));
      if (pass == 0) total += sz;
      else tma_load_1d(buf + (size_t)i * p.dn_piece_bytes, a, sz, bar, pol);
    }
    if (pass == 0) mbar_arrive_expect_tx(bar, total);
  }
}

// One down work item: one row per LPR-lane group (32/LPR rows) against up to
// NTT routes' intermediates; results reduced within each lane group.
template <int WT, int LPR, int NTT>
__device__ __forceinline__ void dn_item(const uint8_t* rowp, bool vrow, int I, int sl, const ActSrc& act,
                                        const int (&rt)[NT], int nt, float (&res)[NT]) {
  float acc[NTT];
#pragma unroll
  for (int t = 0; t < NTT; ++t) acc[t] = 0.f;
  if (vrow) {
    if constexpr (is_float_w(WT)) {
      for (int c = sl; c < I / 8; c += LPR) {
        float wv[8];
        float_row_chunk8<WT>(rowp, c, wv);
#pragma unroll
        for (int t = 0; t < NTT; ++t) {
          if (NTT == 1 || t < nt) {
            const float4* ip = reinterpret_cast<const float4*>(act.xf + (size_t)rt[t] * I + 8 * c);
            const float4 v0 = ip[0], v1 = ip[1];
            acc[t] = fmaf(wv[0], v0.x, acc[t]); acc[t] = fmaf(wv[1], v0.y, acc[t]);
            acc[t] = fmaf(wv[2], v0.z, acc[t]); acc[t] = fmaf(wv[3], v0.w, acc[t]);
            acc[t] = fmaf(wv[4], v1.x, acc[t]); acc[t] = fmaf(wv[5], v1.y, acc[t]);
            acc[t] = fmaf(wv[6], v1.z, acc[t]); acc[t] = fmaf(wv[7], v1.w, acc[t]);
          }
        }
      }
    } else {
      const int nbi = I / 32;
      int b = sl;
      for (; NTT <= 2 && b + LPR < nbi; b += 2 * LPR) {
        ActQ8 a0[NTT], a1[NTT];
#pragma unroll
        for (int t = 0; t < NTT; ++t)
          if (NTT == 1 || t < nt) {
            a0[t] = act_block(act, rt[t], b);
            a1[t] = act_block(act, rt[t], b + LPR);
          }
        accum_q_block<WT, NTT>(rowp, I, b, a0, nt, acc);
        accum_q_block<WT, NTT>(rowp, I, b + LPR, a1, nt, acc);
      }
      for (; b < nbi; b += LPR) {
        ActQ8 a[NTT];
#pragma unroll
        for (int t = 0; t < NTT; ++t)
          if (NTT == 1 || t < nt) a[t] = act_block(act, rt[t], b);
        accum_q_block<WT, NTT>(rowp, I, b, a, nt, acc);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NTT; ++t) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    res[t] = acc[t];
  }
}

}  // namespace qre
