// Routed-expert MoE decode kernels for sm_103a.
//
// One decode pass is three kernels on one stream, chained with programmatic
// dependent launch (PDL):
//
//   k_prep     prep_input: waits for the previous grid, lets the next grid
//              start, zeroes the per-block counters and quantizes the bf16
//              hidden states to q8_1 (FreeToken PR #704, "How it plugs into
//              the CPU executor", prep_input; Strata PR #292,
//              "Summary/Pipeline": q8_1 activations).
//   k_gate_up  gate_up + prep_inter: every CTA groups the routes by expert,
//              takes a cost-balanced run of (expert, i) pairs (gate row i and
//              up row I+i), streams those rows into a ring of shared-memory
//              stages with 1-D TMA bulk copies issued *before* waiting on
//              k_prep, dots them with the q8_1 activations of every token
//              routed to the expert, applies s_gate / s_up in fp32 and
//              SiLU-GLU (FreeToken PR #732, "Design"; Strata PR #292: each
//              global scale multiplies its own projection's fp32 output), and
//              requantizes the intermediate to q8_1 for a quantized down type.
//              A 32-block of the intermediate that straddles CTAs is
//              quantized by the last CTA to finish its part (a counter per
//              block), so work is split at pair granularity.
//   k_down     down + route sum: every CTA owns a run of output rows, streams
//              those rows of every routed expert (prefetched before waiting on
//              k_gate_up), dots them with each route's intermediate, and sums
//              the routes of a token in route order k = 0..K-1 with the routing
//              weight and s_down, writing bf16 with no atomics.
//
// Each selected expert's rows are read from HBM once per pass, whatever the
// number of tokens routed to it.
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

// Named barrier 1 synchronises the consumer warps only (the producer warp
// may already have left).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
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
__device__ int block_exclusive_scan(int* a, int n, int* wsum) {
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

// Group the T*K routes by expert: the distinct valid experts in ascending id
// order become slots; each slot lists its routes in route order.  Reads only
// `ids`.  Every CTA of a kernel computes the same grouping.  Up to 32 routes
// one warp does it with match/shuffle; beyond that the whole block scans.
__device__ void group_routes(const int32_t* ids, int RT, int E, int K, const GroupSmem& g) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x;
  if (RT <= 32) {
    if (warp == 0) {
      int e = (lane < RT) ? ids[lane] : -1;
      const bool valid = (lane < RT) && e >= 0 && e < E;
      const bool bad = (lane < RT) && !valid;
      const int key = valid ? e : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const bool first = valid && (lane == __ffs(peers) - 1);
      int slot = 0, off = 0;
      for (int j = 0; j < 32; ++j) {
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

// ------------------------------------------------------------------ prep

// Load the 32 values of block b (bf16 when kBf16In, else fp32).
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


__global__ void __launch_bounds__(kThreads) k_prep(const __grid_constant__ DecodeParams p, int quantize_x) {
  pdl_wait();                 // the previous grid (and whatever produced x and ids) is complete
  pdl_launch_dependents();    // k_gate_up may now start its id-dependent prologue
  const int gtid = blockIdx.x * kThreads + threadIdx.x;
  const int nthr = gridDim.x * kThreads;
  for (int i = gtid; i < p.cnt_len; i += nthr) p.cnt[i] = 0u;
  if (!quantize_x) return;
  const int nb = p.H / 32;
  for (int b = gtid; b < p.T * nb; b += nthr) {
    float v[32];
    load_block32<true>(p.x, b, v);
    uint32_t qw[8];
    float d;
    int sum;
    q8_1_quantize_block(v, qw, d, sum);
    uint4* qd = reinterpret_cast<uint4*>(p.xq + (size_t)b * 32);
    qd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    qd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    p.xd[b] = f16_bits_to_f32(f32_to_f16_bits_rn(d));
    p.xsum[b] = sum;
    p.xsh[b] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
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
__device__ void pair_at_cost(long long target, const int* slot_off, int S, int I, int w0, int& u, int& i) {
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

// floor(W * c / G) for the CTA boundaries, through fp64 (exact below 2^53).
__device__ __forceinline__ long long cost_cut(long long W, int c, int G) {
  return (long long)floor((double)W * (double)c / (double)G);
}

__device__ __forceinline__ const uint8_t* align16_down(const uint8_t* a) {
  return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15));
}
__device__ __forceinline__ uint32_t round16(uint32_t v) { return (v + 15u) & ~15u; }

__device__ void issue_gu_stage(const DecodeParams& p, uint8_t* buf, uint64_t* bar, int e, int i0, int n,
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
__device__ void copy_to_smem(void* dst, const void* src, size_t bytes) {
  const int tid = threadIdx.x;
  if ((bytes & 15) == 0) {
    const size_t n = bytes / 16;
    const int4* s = static_cast<const int4*>(src);
    int4* d = static_cast<int4*>(dst);
    for (size_t i = tid; i < n; i += 4 * kConsumerThreads) {
      int4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * kConsumerThreads < n) v[j] = __ldcg(s + i + j * kConsumerThreads);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * kConsumerThreads < n) d[i + j * kConsumerThreads] = v[j];
    }
  } else {
    const size_t n = bytes / 4;
    const int* s = static_cast<const int*>(src);
    int* d = static_cast<int*>(dst);
    for (size_t i = tid; i < n; i += kConsumerThreads) d[i] = __ldcg(s + i);
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
#pragma unroll
    for (int t = 0; t < NTT; ++t) {
      if (NTT == 1 || t < nt) {
        int d0, d1;
        nvfp4_int_dots(pos, neg, a[t].q, d0, d1);
        acc[t] += a[t].d * 0.5f * (s.x * (float)d0 + s.y * (float)d1);
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
  } else {  // W_Q8_0
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
  if constexpr (WT == W_BF16) {
    for (int c = b0 + lane; c < b1; c += 32) {
      float wg[8], wu[8];
      bf16x8_to_f32(lds128(grow + 16 * c), wg);
      bf16x8_to_f32(lds128(urow + 16 * c), wu);
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
__device__ __forceinline__ float silu_glu(float g, float u) { return __fdividef(g, 1.0f + expf(-g)) * u; }

// Quantize `nblk` 32-value blocks (row-major values from `src`) into q8_1
// planes in shared memory -- codes q[32*b + i], scales d[b] (fp16 values as
// fp32), code sums sm[b] -- one block per consumer thread.  When `ids` is
// given, blocks of routes (rows of `blocks_per_row` blocks) with an invalid
// expert id are skipped.  With `mirror`, the blocks also go to the workspace
// planes (wq, wd, wsum, wsh) for inspection.
template <bool kBf16In>
__device__ void quantize_blocks_to_smem(const void* src, int nblk, const int32_t* ids, int E, int blocks_per_row,
                                        int8_t* q, float* d, int* sm, bool mirror, int8_t* wq, float* wd, int* wsum,
                                        uint16_t* wsh) {
  for (int b = threadIdx.x; b < nblk; b += kConsumerThreads) {
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

// MAXNT = 1 (batches of up to two tokens): the x quantizer runs inside this
// kernel, which waits for the previous grid before touching ids, and the
// intermediate is requantized by k_down.  MAXNT = 4: k_prep quantizes x and
// has already waited, so ids are read before this kernel waits, and the
// intermediate is requantized here by the last CTA to finish each block.
// Launch bounds keep registers low enough for a k_down CTA to share the SM.
template <int WT, int MAXNT>
__global__ void __launch_bounds__(kDecodeThreads, MAXNT == 1 ? 2 : 1) k_gate_up(const __grid_constant__ DecodeParams p) {
  constexpr bool kFused = (MAXNT == 1);
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RT = p.T * p.K;
  const int NS = p.gu_nstage;
  constexpr int kPart = kConsumerWarps * NT * 2;

  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * p.gu_stage_bytes);
  uint64_t* empty = full + NS;
  float* part = reinterpret_cast<float*>(empty + NS);                    // [NS][kPart]
  int* pcnt = reinterpret_cast<int*>(part + (size_t)NS * kPart);         // [NS]
  uint8_t* actm = reinterpret_cast<uint8_t*>(pcnt + NS);
  actm += (16 - (reinterpret_cast<uintptr_t>(actm) & 15)) & 15;
  GroupSmem g = carve_group(actm + p.gu_act_bytes, p.E, RT);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
      pcnt[s] = 0;
    }
    fence_mbar_init();
  }
  if constexpr (kFused) pdl_wait();   // ids and x may come from the previous grid
  group_routes(p.ids, RT, p.E, p.K, g);
  const int S = g.misc[0];
  if (tid == 0) {
    int ub, ib, ue, ie;
    if constexpr (kFused) {
      // one or two tokens: every expert costs about the same per pair, so
      // split the pairs evenly (32-bit arithmetic)
      const unsigned P = (unsigned)S * (unsigned)p.I;
      const unsigned lo = (unsigned)((unsigned long long)P * blockIdx.x / gridDim.x);
      const unsigned hi = (unsigned)((unsigned long long)P * (blockIdx.x + 1) / gridDim.x);
      ub = lo / p.I; ib = lo - ub * p.I;
      ue = hi / p.I; ie = hi - ue * p.I;
    } else {
      long long W = 0;
      for (int s = 0; s < S; ++s) W += (long long)(p.w0 + g.slot_off[s + 1] - g.slot_off[s]) * p.I;
      const long long lo = cost_cut(W, blockIdx.x, gridDim.x), hi = cost_cut(W, blockIdx.x + 1, gridDim.x);
      pair_at_cost(lo, g.slot_off, S, p.I, p.w0, ub, ib);
      pair_at_cost(hi, g.slot_off, S, p.I, p.w0, ue, ie);
    }
    g.misc[2] = ub; g.misc[3] = ib; g.misc[4] = ue; g.misc[5] = ie;
    g.misc[6] = 0;
    g.misc[7] = 0;
    if (blockIdx.x == 0 && g.misc[1]) atomicOr(p.err, kErrBadId);
  }
  __syncthreads();
  const int ub = g.misc[2], ib = g.misc[3], ue = g.misc[4], ie = g.misc[5];

  if (warp == kProducerWarp) {
    // TMA producer: streams the CTA's pairs through the NS-deep ring.
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      PairCursor pc{ub, ib};
      int buf = 0;
      uint32_t eph = 0;
      bool wrapped = false;
      for (;;) {
        int su, si, sn;
        if (!next_gu_stage(pc, ue, ie, p.I, p.ps, su, si, sn)) break;
        if (wrapped) {
          if (!mbar_wait_bounded(&empty[buf], eph, kWaitLimit)) {
            g.misc[6] = 1;
            break;
          }
          fence_proxy_async_smem();
        }
        issue_gu_stage(p, stages + (size_t)buf * p.gu_stage_bytes, &full[buf], g.slot_e[su], si, sn, pol);
        atomicAdd(&g.misc[7], 1);
        if (++buf == NS) {
          buf = 0;
          if (wrapped) eph ^= 1u;
          wrapped = true;
        }
      }
    }
    pdl_launch_dependents();
    return;
  }

  if constexpr (!kFused) pdl_wait();  // k_prep complete: activations and zeroed counters are visible
  pdl_launch_dependents();

  // Scale pairs of the slots (off the producer's path).
  for (int sl = tid; sl < S; sl += kConsumerThreads) {
    const int e = g.slot_e[sl];
    g.sscale[3 * sl + 0] = __ldg(p.scales + 4 * e + 0);
    g.sscale[3 * sl + 1] = __ldg(p.scales + 4 * e + 1);
  }
  // Activations: in shared memory when they fit, else read from the workspace.
  ActSrc act;
  act.n = p.H;
  act.xb = p.x;
  if (WT == W_BF16) {
    if (p.gu_act_smem) {
      copy_to_smem(actm, p.x, 2 * (size_t)p.T * p.H);
      act.xb = reinterpret_cast<const uint16_t*>(actm);
    }
  } else if (p.gu_act_smem) {
    const int nbh = p.H / 32;
    int8_t* q = reinterpret_cast<int8_t*>(actm);
    float* d = reinterpret_cast<float*>(actm + (size_t)p.T * p.H);
    int* sm = reinterpret_cast<int*>(d + (size_t)p.T * nbh);
    if constexpr (kFused) {
      quantize_blocks_to_smem<true>(p.x, p.T * nbh, nullptr, p.E, nbh, q, d, sm, blockIdx.x == 0, p.xq, p.xd,
                                    p.xsum, p.xsh);
    } else {
      copy_to_smem(q, p.xq, (size_t)p.T * p.H);
      copy_to_smem(d, p.xd, 4 * (size_t)p.T * nbh);
      copy_to_smem(sm, p.xsum, 4 * (size_t)p.T * nbh);
    }
    act.q = q; act.d = d; act.s = sm;
  } else {
    act.q = p.xq; act.d = p.xd; act.s = p.xsum;
  }
  consumer_sync();

  const bool requant = !kFused && (p.dn_type != W_BF16);
  const int nb = (WT == W_BF16) ? p.H / 8 : p.H / 32;   // blocks (8 values for BF16, 32 otherwise)
  const int max_ks = max(1, nb / 32);
  const int cw = warp;                                  // consumer warp 0..7
  const size_t rbg = (size_t)p.rb_gu;

  PairCursor cc{ub, ib};
  int rot = 0;   // rotates which consumer warp takes a stage's first pair
  int s = 0, buf = 0;
  uint32_t fph = 0;
  for (;; ++s) {
    int su, si, sn;
    if (!next_gu_stage(cc, ue, ie, p.I, p.ps, su, si, sn)) break;
    const uint8_t* sbuf = stages + (size_t)buf * p.gu_stage_bytes;
    const int e = g.slot_e[su];
    const uint8_t* gsrc = p.gu_bank + ((size_t)e * 2 * p.I + si) * rbg;
    const uint8_t* usrc = gsrc + (size_t)p.I * rbg;
    const uint8_t* gbase = sbuf + (gsrc - align16_down(gsrc));
    const uint8_t* ubase = sbuf + p.gu_up_off + (usrc - align16_down(usrc));
    const int roff = g.slot_off[su];
    const int Tu = g.slot_off[su + 1] - roff;
    const int nch = (Tu + MAXNT - 1) / MAXNT;
    const int base_items = sn * nch;
    const int ks_n = base_items < kConsumerWarps ? max(1, min(kConsumerWarps / base_items, max_ks)) : 1;
    const float sg = g.sscale[3 * su + 0], su_ = g.sscale[3 * su + 1];
    float* pbuf = part + (size_t)buf * kPart;
    // Every consumer waits for the stage, work or not: that orders its use of
    // pcnt[buf] after the previous user of this buffer reset it.
    if (!mbar_wait_bounded(&full[buf], fph, kWaitLimit)) {
      g.misc[6] = 1;
      break;
    }
    if (ks_n == 1) {
      // whole rows per item: pairs round-robin over the warps, route chunks inside
      for (int pi = (cw - rot) & (kConsumerWarps - 1); pi < sn; pi += kConsumerWarps) {
        const uint8_t* grow = gbase + (size_t)pi * rbg;
        const uint8_t* urow = ubase + (size_t)pi * rbg;
        for (int c0 = 0; c0 < Tu; c0 += MAXNT) {
          const int nt = min(MAXNT, Tu - c0);
          int tok[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) tok[t] = (t < nt) ? (int)g.rtok[roff + c0 + t] : 0;
          float ag[NT], au[NT];
          if (MAXNT == 1 || nt == 1) gu_item<WT, 1>(grow, urow, p.H, 0, nb, lane, act, tok, nt, ag, au);
          else if (nt == 2) gu_item<WT, 2>(grow, urow, p.H, 0, nb, lane, act, tok, nt, ag, au);
          else gu_item<WT, (MAXNT > 1 ? 4 : 1)>(grow, urow, p.H, 0, nb, lane, act, tok, nt, ag, au);
          if (lane < nt) {
            float gv = ag[0], uv = au[0];
#pragma unroll
            for (int t = 1; t < NT; ++t)
              if (lane == t) { gv = ag[t]; uv = au[t]; }
            const int r = g.routes[roff + c0 + lane];
            p.inter[(size_t)r * p.I + si + pi] = silu_glu(gv * sg, uv * su_);
          }
        }
      }
      rot = (rot + sn) & (kConsumerWarps - 1);
    } else {
      // few (pair, chunk) items: each also split along K; at most one item per warp
      const int it = cw;
      if (it < base_items * ks_n) {
        const int ks = it / base_items, rem = it - ks * base_items;
        const int ch = rem / sn, pi = rem - ch * sn;
        const int nt = min(MAXNT, Tu - ch * MAXNT);
        int tok[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) tok[t] = (t < nt) ? (int)g.rtok[roff + ch * MAXNT + t] : 0;
        const int b0 = nb * ks / ks_n, b1 = nb * (ks + 1) / ks_n;
        const uint8_t* grow = gbase + (size_t)pi * rbg;
        const uint8_t* urow = ubase + (size_t)pi * rbg;
        float ag[NT], au[NT];
        if (MAXNT == 1 || nt == 1) gu_item<WT, 1>(grow, urow, p.H, b0, b1, lane, act, tok, nt, ag, au);
        else if (nt == 2) gu_item<WT, 2>(grow, urow, p.H, b0, b1, lane, act, tok, nt, ag, au);
        else gu_item<WT, (MAXNT > 1 ? 4 : 1)>(grow, urow, p.H, b0, b1, lane, act, tok, nt, ag, au);
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            pbuf[(it * NT + t) * 2 + 0] = ag[t];
            pbuf[(it * NT + t) * 2 + 1] = au[t];
          }
        }
      }
      // The last consumer warp to finish the stage sums the partials in
      // K-slice order and applies the epilogue.
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = (atomicAdd(&pcnt[buf], 1) == kConsumerWarps - 1);
        if (last) __threadfence_block();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        for (int idx = lane; idx < Tu * sn; idx += 32) {
          const int ri = idx / sn, pi = idx - ri * sn;
          const int ch = ri / MAXNT, t = ri - ch * MAXNT;
          float hg = 0.f, hu = 0.f;
          for (int ks = 0; ks < ks_n; ++ks) {
            const int it2 = ks * base_items + ch * sn + pi;
            hg += pbuf[(it2 * NT + t) * 2 + 0];
            hu += pbuf[(it2 * NT + t) * 2 + 1];
          }
          const int r = g.routes[roff + ri];
          p.inter[(size_t)r * p.I + si + pi] = silu_glu(hg * sg, hu * su_);
        }
        __syncwarp();
        if (lane == 0) pcnt[buf] = 0;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[buf]);
    if (++buf == NS) {
      buf = 0;
      fph ^= 1u;
    }
  }

  consumer_sync();
  if (g.misc[6]) {  // a bounded wait ran out: drain what is in flight (bounded), flag, leave
    if (tid == 0) {
      const int issued = g.misc[7];
      for (int q = s; q < issued; ++q) mbar_wait_bounded(&full[q % NS], (uint32_t)((q / NS) & 1), kWaitLimit);
      atomicOr(p.err, kErrTimeout);
    }
    return;
  }
  if (!requant) return;

  // prep_inter for batches of three tokens or more: q8_1 requantization of
  // each completed 32-block of the intermediate.  Each CTA adds the pairs it
  // wrote to the block's counter; the CTA that completes a block (counter
  // reaches 32) quantizes it for every route of that expert.
  const int nbi = p.I / 32;
  int j = 0;
  for (int u = ub; u <= ue && u < S; ++u) {
    const int a0 = (u == ub) ? ib : 0;
    const int a1 = (u == ue) ? ie : p.I;
    if (a1 <= a0) continue;
    for (int blk = a0 / 32; blk <= (a1 - 1) / 32; ++blk, ++j) {
      if ((j % kConsumerWarps) != cw) continue;
      const int c = min(a1, 32 * (blk + 1)) - max(a0, 32 * blk);
      unsigned old = 0;
      if (lane == 0) {
        __threadfence();
        old = atomicAdd(&p.cnt[u * nbi + blk], (unsigned)c);
        __threadfence();
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old + (unsigned)c != 32u) continue;
      const int roff = g.slot_off[u], Tu = g.slot_off[u + 1] - roff;
      __threadfence();
      for (int ri = lane; ri < Tu; ri += 32) {
        const int r = g.routes[roff + ri];
        const int b = r * nbi + blk;
        float v[32];
        load_block32<false>(p.inter, b, v);
        uint32_t qw[8];
        float d;
        int sum;
        q8_1_quantize_block(v, qw, d, sum);
        uint4* qd = reinterpret_cast<uint4*>(p.iq + (size_t)b * 32);
        qd[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        qd[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
        p.id[b] = f16_bits_to_f32(f32_to_f16_bits_rn(d));
        p.isum[b] = sum;
        p.ish[b] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
      }
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

__device__ void issue_dn_stage(const DecodeParams& p, uint8_t* buf, uint64_t* bar, const GroupSmem& g,
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
    if constexpr (WT == W_BF16) {
      for (int c = sl; c < I / 8; c += LPR) {
        float wv[8];
        bf16x8_to_f32(lds128(rowp + 16 * c), wv);
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

// MAXNT = 1 (batches of up to two tokens): this kernel requantizes the fp32
// intermediate into shared memory itself (prep_inter) right after waiting.
template <int WT, int LPR, int MAXNT>
__global__ void __launch_bounds__(kDecodeThreads, MAXNT == 1 ? 2 : 1) k_down(const __grid_constant__ DecodeParams p) {
  constexpr bool kFused = (MAXNT == 1);
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RT = p.T * p.K;
  const int NS = p.dn_nstage;
  constexpr int RPI = 32 / LPR;   // rows per work item (one per lane group)

  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * p.dn_stage_bytes);
  uint64_t* empty = full + NS;
  float* ysm = reinterpret_cast<float*>(empty + NS);
  uint8_t* actm = reinterpret_cast<uint8_t*>(ysm + (size_t)RT * p.dn_rows_max);
  actm += (16 - (reinterpret_cast<uintptr_t>(actm) & 15)) & 15;
  GroupSmem g = carve_group(actm + p.dn_act_bytes, p.E, RT);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  // ids were complete before k_gate_up passed its own wait, so they may be
  // read before this kernel waits.
  group_routes(p.ids, RT, p.E, p.K, g);
  const int S = g.misc[0];
  const int j0 = (int)((long long)p.H * blockIdx.x / gridDim.x);
  const int j1 = (int)((long long)p.H * (blockIdx.x + 1) / gridDim.x);
  const int nj = j1 - j0;
  const int sps = p.dn_slots_per_stage, rs = p.dn_rs;
  const int ngrp = (S + sps - 1) / sps;
  const int nst = (S > 0 && nj > 0) ? ((nj + rs - 1) / rs) * ngrp : 0;
  if (tid == 0) {
    g.misc[6] = 0;
    g.misc[7] = 0;
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int buf = 0;
      uint32_t eph = 0;
      bool wrapped = false;
      for (int k = 0; k < nst; ++k) {
        if (wrapped) {
          if (!mbar_wait_bounded(&empty[buf], eph, kWaitLimit)) {
            g.misc[6] = 1;
            break;
          }
          fence_proxy_async_smem();
        }
        issue_dn_stage(p, stages + (size_t)buf * p.dn_stage_bytes, &full[buf], g, down_stage(k, S, nj, rs, sps), j0,
                       pol);
        atomicAdd(&g.misc[7], 1);
        if (++buf == NS) {
          buf = 0;
          if (wrapped) eph ^= 1u;
          wrapped = true;
        }
      }
    }
    pdl_launch_dependents();
    return;
  }

  pdl_launch_dependents();
  pdl_wait();  // k_gate_up complete: the intermediate is visible

  ActSrc act;
  act.n = p.I;
  act.xf = p.inter;
  if (WT == W_BF16) {
    if (p.dn_act_smem) {
      copy_to_smem(actm, p.inter, 4 * (size_t)RT * p.I);
      act.xf = reinterpret_cast<const float*>(actm);
    }
  } else if (p.dn_act_smem) {
    const int nbi = p.I / 32;
    int8_t* q = reinterpret_cast<int8_t*>(actm);
    float* d = reinterpret_cast<float*>(actm + (size_t)RT * p.I);
    int* sm = reinterpret_cast<int*>(d + (size_t)RT * nbi);
    if constexpr (kFused) {
      // prep_inter: fp32 intermediate -> q8_1 (routes with a bad id skipped);
      // CTA 0 mirrors the blocks to the workspace for inspection.
      quantize_blocks_to_smem<false>(p.inter, RT * nbi, p.ids, p.E, nbi, q, d, sm, blockIdx.x == 0, p.iq, p.id,
                                     p.isum, p.ish);
    } else {
      copy_to_smem(q, p.iq, (size_t)RT * p.I);
      copy_to_smem(d, p.id, 4 * (size_t)RT * nbi);
      copy_to_smem(sm, p.isum, 4 * (size_t)RT * nbi);
    }
    act.q = q; act.d = d; act.s = sm;
  } else {
    act.q = p.iq; act.d = p.id; act.s = p.isum;
  }
  consumer_sync();

  const int cw = warp;
  const int grp = lane / LPR, sl = lane % LPR;
  const size_t rbd = (size_t)p.rb_dn;
  int rot = 0;
  int k = 0, buf = 0;
  uint32_t fph = 0;
  for (; k < nst; ++k) {
    const uint8_t* sbuf = stages + (size_t)buf * p.dn_stage_bytes;
    const DownStage st = down_stage(k, S, nj, rs, sps);
    const int nq = (st.nr + RPI - 1) / RPI;
    if (!mbar_wait_bounded(&full[buf], fph, kWaitLimit)) {
      g.misc[6] = 1;
      break;
    }
    // (slot, row group) items round-robin over the warps, route chunks inside
    for (int i = 0; i < st.ns; ++i) {
      const int u = st.u0 + i;
      const int roff = g.slot_off[u];
      const int Tu = g.slot_off[u + 1] - roff;
      const int e = g.slot_e[u];
      const uint8_t* src = p.dn_bank + ((size_t)e * p.H + j0 + st.js) * rbd;
      const uint8_t* piece = sbuf + (size_t)i * p.dn_piece_bytes + (src - align16_down(src));
      for (int q = (cw - rot) & (kConsumerWarps - 1); q < nq; q += kConsumerWarps) {
        const int row = q * RPI + grp;
        const bool vrow = row < st.nr;
        const uint8_t* rowp = piece + (size_t)(vrow ? row : 0) * rbd;
        for (int c0 = 0; c0 < Tu; c0 += MAXNT) {
          const int nt = min(MAXNT, Tu - c0);
          int rt[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) rt[t] = (t < nt) ? (int)g.routes[roff + c0 + t] : 0;
          float res[NT];
          if (MAXNT == 1 || nt == 1) dn_item<WT, LPR, 1>(rowp, vrow, p.I, sl, act, rt, nt, res);
          else if (nt == 2) dn_item<WT, LPR, 2>(rowp, vrow, p.I, sl, act, rt, nt, res);
          else dn_item<WT, LPR, (MAXNT > 1 ? 4 : 1)>(rowp, vrow, p.I, sl, act, rt, nt, res);
          if (vrow && sl < nt) {
            float v = res[0];
            int r = rt[0];
#pragma unroll
            for (int t = 1; t < NT; ++t)
              if (sl == t) { v = res[t]; r = rt[t]; }
            ysm[(size_t)r * p.dn_rows_max + st.js + row] = v;
          }
        }
      }
      rot = (rot + nq) & (kConsumerWarps - 1);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[buf]);
    if (++buf == NS) {
      buf = 0;
      fph ^= 1u;
    }
  }
  consumer_sync();
  if (g.misc[6]) {
    if (tid == 0) {
      const int issued = g.misc[7];
      for (int q = k; q < issued; ++q) mbar_wait_bounded(&full[q % NS], (uint32_t)((q / NS) & 1), kWaitLimit);
      atomicOr(p.err, kErrTimeout);
    }
    return;
  }
  // Route sum in route order k = 0..K-1, then one rounding to bf16.
  for (int idx = tid; idx < p.T * nj; idx += kConsumerThreads) {
    const int t = idx / nj, jj = idx - t * nj;
    float acc = 0.f;
    for (int kk = 0; kk < p.K; ++kk) {
      const int r = t * p.K + kk;
      const int e = p.ids[r];
      if (e < 0 || e >= p.E) continue;
      acc += ysm[(size_t)r * p.dn_rows_max + jj] * (__ldg(p.scales + 4 * e + 2) * __ldg(p.w + r));
    }
    p.out[(size_t)t * p.H + j0 + jj] = (uint16_t)f32_to_bf16_bits_rn(acc);
  }
}

// ------------------------------------------------------------------ launch

static int g_sm_count = 0;
int sm_count() {
  if (g_sm_count == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (g_sm_count <= 0) g_sm_count = 1;
  }
  return g_sm_count;
}

size_t gate_up_smem_bytes(const DecodeParams& p) {
  const int RT = p.T * p.K;
  return (size_t)p.gu_nstage * p.gu_stage_bytes + 16 * (size_t)p.gu_nstage +
         sizeof(float) * (size_t)p.gu_nstage * kConsumerWarps * NT * 2 + sizeof(int) * (size_t)p.gu_nstage + 16 +
         (size_t)p.gu_act_bytes + group_smem_bytes(p.E, RT);
}

size_t down_smem_bytes(const DecodeParams& p) {
  const int RT = p.T * p.K;
  return (size_t)p.dn_nstage * p.dn_stage_bytes + 16 * (size_t)p.dn_nstage +
         sizeof(float) * (size_t)RT * p.dn_rows_max + 16 + (size_t)p.dn_act_bytes + group_smem_bytes(p.E, RT);
}

template <typename K>
static cudaError_t launch_pdl(K kernel, int grid, size_t smem, cudaStream_t stream, const DecodeParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_prep(const DecodeParams& p, cudaStream_t stream) {
  const int quantize_x = (p.gu_type != W_BF16) ? 1 : 0;
  const int work = quantize_x ? (p.T * (p.H / 32) + kThreads - 1) / kThreads : 1;
  const int cntb = (p.cnt_len + kThreads - 1) / kThreads;
  int grid = work > cntb ? work : cntb;
  if (grid > 4 * sm_count()) grid = 4 * sm_count();
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_prep, p, quantize_x);
}

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int WT, int MAXNT>
static cudaError_t launch_gu_t(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_smem(k_gate_up<WT, MAXNT>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_gate_up<WT, MAXNT>, p.g_gu, smem, stream, p);
}

template <int WT>
static cudaError_t launch_gu_w(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  return p.maxnt == 1 ? launch_gu_t<WT, 1>(p, smem, stream) : launch_gu_t<WT, 4>(p, smem, stream);
}

cudaError_t launch_gate_up(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = gate_up_smem_bytes(p);
  switch (p.gu_type) {
    case W_NVFP4:
      if (p.rb_gu % 16 != 0) return launch_gu_w<W_NVFP4_U>(p, smem, stream);
      return launch_gu_w<W_NVFP4>(p, smem, stream);
    case W_Q4_K: return launch_gu_w<W_Q4_K>(p, smem, stream);
    case W_Q8_0: return launch_gu_w<W_Q8_0>(p, smem, stream);
    default: return launch_gu_w<W_BF16>(p, smem, stream);
  }
}

template <int WT, int LPR, int MAXNT>
static cudaError_t launch_dn_t(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_smem(k_down<WT, LPR, MAXNT>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_down<WT, LPR, MAXNT>, p.g_dn, smem, stream, p);
}

template <int WT, int LPR>
static cudaError_t launch_dn_w(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  return p.maxnt == 1 ? launch_dn_t<WT, LPR, 1>(p, smem, stream) : launch_dn_t<WT, LPR, 4>(p, smem, stream);
}

cudaError_t launch_down(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = down_smem_bytes(p);
  switch (p.dn_type) {
    case W_NVFP4:
      if (p.rb_dn % 16 != 0) return launch_dn_w<W_NVFP4_U, 8>(p, smem, stream);
      return launch_dn_w<W_NVFP4, 8>(p, smem, stream);
    case W_Q4_K: return launch_dn_w<W_Q4_K, 8>(p, smem, stream);
    case W_Q8_0: return launch_dn_w<W_Q8_0, 8>(p, smem, stream);
    default: return launch_dn_w<W_BF16, 16>(p, smem, stream);
  }
}

// ------------------------------------------------------------------ test hooks

__global__ void k_quantize_blocks(const float* x, int64_t nblocks, uint8_t* out) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = x[b * 32 + i];
  uint32_t qw[8];
  float d;
  int sum;
  q8_1_quantize_block(v, qw, d, sum);
  uint32_t* blk = reinterpret_cast<uint32_t*>(out + 36 * b);
  blk[0] = f32_to_f16_bits_rn(d) | (f32_to_f16_bits_rn(d * (float)sum) << 16);
#pragma unroll
  for (int w = 0; w < 8; ++w) blk[1 + w] = qw[w];
}

cudaError_t launch_quantize_q8_1_blocks(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  const int64_t nb = n / 32;
  if (nb == 0) return cudaSuccess;
  const int64_t grid = (nb + 127) / 128;
  k_quantize_blocks<<<(unsigned)grid, 128, 0, stream>>>(x, nb, out);
  return cudaGetLastError();
}

__device__ __forceinline__ ActQ8 act_from_block(const uint8_t* blk) {
  ActQ8 a;
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(blk + 4);
#pragma unroll
  for (int i = 0; i < 8; ++i) a.q[i] = (int)qw[i];
  a.d = f16_bits_to_f32((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
  a.sum = 0;
  return a;
}

__global__ void k_block_dots(int type, const uint8_t* rows, int nrows, int k, const uint8_t* act, int32_t* out) {
  const int nb = k / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)nrows * nb) return;
  const int r = (int)(idx / nb), b = (int)(idx % nb);
  const int rb = row_bytes_of(type, k);
  const uint8_t* row = rows + (size_t)r * rb;
  const ActQ8 a = act_from_block(act + 36 * (size_t)b);
  if (type == W_NVFP4) {
    uint32_t pos[8], neg[8];
    float2 s;
    if ((rb & 15) == 0) nvfp4_decode<true>(row, k, b, pos, neg, s);
    else nvfp4_decode<false>(row, k, b, pos, neg, s);
    int d0, d1;
    nvfp4_int_dots(pos, neg, a.q, d0, d1);
    out[(size_t)r * (k / 16) + 2 * b] = d0;
    out[(size_t)r * (k / 16) + 2 * b + 1] = d1;
  } else if (type == W_Q4_K) {
    int nib[8];
    float dsc, dmm;
    q4k_decode(row, b, nib, dsc, dmm);
    out[(size_t)r * nb + b] = int_dot8(nib, a.q);
  } else {
    int wq[8];
    float d;
    q8_0_decode(row, b, wq, d);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q);
  }
}

cudaError_t launch_block_dots(int type, const uint8_t* rows, int nrows, int k, const uint8_t* act, int32_t* out,
                              cudaStream_t stream) {
  const int64_t n = (int64_t)nrows * (k / 32);
  if (n == 0) return cudaSuccess;
  k_block_dots<<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(type, rows, nrows, k, act, out);
  return cudaGetLastError();
}

__global__ void k_export_q8(const int8_t* q, const float* d, const uint16_t* s, int64_t nblocks, uint8_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblocks * 36) return;
  const int64_t b = i / 36;
  const int o = (int)(i % 36);
  uint8_t v;
  if (o < 2) {
    const uint32_t dh = f32_to_f16_bits_rn(d[b]);
    v = (uint8_t)((o == 0) ? (dh & 0xFFu) : (dh >> 8));
  } else if (o < 4) {
    v = (o == 2) ? (s[b] & 0xFF) : (s[b] >> 8);
  } else {
    v = (uint8_t)q[b * 32 + (o - 4)];
  }
  out[i] = v;
}

cudaError_t launch_export_q8(const int8_t* q, const float* d, const uint16_t* s, int64_t nblocks, uint8_t* out,
                             cudaStream_t stream) {
  const int64_t n = nblocks * 36;
  if (n == 0) return cudaSuccess;
  k_export_q8<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(q, d, s, nblocks, out);
  return cudaGetLastError();
}

}  // namespace qre
