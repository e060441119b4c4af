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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int NT = 4;                       // routes per work item held in registers
constexpr uint32_t kWaitLimit = 1u << 24;   // polls of a TMA barrier before giving up
constexpr uint32_t kErrBadId = 1u, kErrTimeout = 2u;

// ------------------------------------------------------------------ grouping

struct GroupSmem {
  int* slot_of;     // [E]   expert -> slot (valid for experts that are routed to)
  int* slot_e;      // [S]   slot -> expert, ascending expert id
  int* slot_off;    // [S+1] start of each slot's routes in `routes`
  int* cursor;      // [S]
  int* misc;        // [8]   0: slot count, 1: bad id seen, 2..5: pair range, 6: abort flag
  int* wsum;        // [kWarps + 1]
  int16_t* routes;  // [T*K] route indices t*K+k grouped by slot, route order inside a slot
};

__host__ __device__ inline size_t group_smem_bytes(int E, int RT) {
  const int S = E < RT ? E : RT;
  return sizeof(int) * (size_t)(E + S + (S + 1) + S + 8 + (kWarps + 1)) + sizeof(int16_t) * (size_t)RT;
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
  g.wsum = p; p += kWarps + 1;
  g.routes = reinterpret_cast<int16_t*>(p);
  return g;
}

// Exclusive prefix sum of a[0..n) in place (block-wide); returns the total.
__device__ int block_exclusive_scan(int* a, int n, int* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kThreads - 1) / kThreads;
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
    const int v = (lane < kWarps) ? wsum[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < kWarps) wsum[lane] = inc - v;
    if (lane == kWarps - 1) wsum[kWarps] = inc;
  }
  __syncthreads();
  int run = wsum[warp] + incl - local;
  for (int i = b0; i < b1; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  const int total = wsum[kWarps];
  __syncthreads();
  return total;
}

// Group the T*K routes by expert: the distinct valid experts in ascending id
// order become slots; each slot lists its routes in route order.  Reads only
// `ids`.  Every CTA of a kernel computes the same grouping.
__device__ void group_routes(const int32_t* ids, int RT, int E, const GroupSmem& g) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kThreads) g.slot_of[e] = 0;
  if (tid == 0) g.misc[1] = 0;
  __syncthreads();
  for (int r = tid; r < RT; r += kThreads) {
    const int e = ids[r];
    if (e >= 0 && e < E) g.slot_of[e] = 1;
    else g.misc[1] = 1;
  }
  __syncthreads();
  const int S = block_exclusive_scan(g.slot_of, E, g.wsum);
  for (int e = tid; e < E; e += kThreads) {
    const int nxt = (e + 1 < E) ? g.slot_of[e + 1] : S;
    if (nxt != g.slot_of[e]) g.slot_e[g.slot_of[e]] = e;
  }
  for (int s = tid; s < S; s += kThreads) g.cursor[s] = 0;
  __syncthreads();
  for (int r = tid; r < RT; r += kThreads) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&g.cursor[g.slot_of[e]], 1);
  }
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) g.slot_off[s] = g.cursor[s];
  __syncthreads();
  const int tot = block_exclusive_scan(g.slot_off, S, g.wsum);
  if (tid == 0) g.slot_off[S] = tot;
  for (int s = tid; s < S; s += kThreads) g.cursor[s] = g.slot_off[s];
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
      if (s >= 0) g.routes[g.cursor[s] + rank] = (int16_t)r;
      __syncwarp();
      if (s >= 0 && rank == 0) g.cursor[s] += __popc(peers);
      __syncwarp();
    }
  }
  if (tid == 0) g.misc[0] = S;
  __syncthreads();
}

// ------------------------------------------------------------------ prep

__global__ void __launch_bounds__(kThreads) k_prep(const __grid_constant__ DecodeParams p, int quantize_x) {
  pdl_wait();                 // the previous grid (and whatever produced x and ids) is complete
  pdl_launch_dependents();    // k_gate_up may now start its id-dependent prologue
  const int gtid = blockIdx.x * kThreads + threadIdx.x;
  const int nthr = gridDim.x * kThreads;
  for (int i = gtid; i < p.cnt_len; i += nthr) p.cnt[i] = 0u;
  if (!quantize_x) return;
  const int lane = threadIdx.x & 31;
  const int nb = p.H / 32;
  const int nwarps = nthr / 32;
  for (int wb = gtid / 32; wb < p.T * nb; wb += nwarps) {
    const int t = wb / nb, b = wb % nb;
    const size_t off = (size_t)t * p.H + 32 * (size_t)b + lane;
    const float v = __uint_as_float((uint32_t)p.x[off] << 16);
    int q, sum;
    float d;
    q8_1_quantize_warp(v, q, d, sum);
    p.xq[off] = (int8_t)q;
    if (lane == 0) {
      const size_t bi = (size_t)t * nb + b;
      p.xd[bi] = f16_bits_to_f32(f32_to_f16_bits_rn(d));
      p.xsum[bi] = sum;
      p.xsh[bi] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
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
__device__ void pair_at_cost(long long target, const int* slot_off, int S, int I, int w0, int& u, int& i) {
  long long c = 0;
  for (u = 0; u < S; ++u) {
    const long long cs = w0 + (slot_off[u + 1] - slot_off[u]);
    const long long span = cs * I;
    if (c + span > target) {
      const long long rem = target - c;
      i = rem <= 0 ? 0 : (int)((rem + cs - 1) / cs);
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

// Accumulate one 32-value block b of a quantized row into acc[0..nt).
template <int WT>
__device__ __forceinline__ void accum_q_block(const uint8_t* row, int k, int b, const ActQ8 (&a)[NT], int nt,
                                              float (&acc)[NT]) {
  if constexpr (WT == W_NVFP4) {
    uint32_t pos[8], neg[8];
    float2 s;
    nvfp4_decode(row, k, b, pos, neg, s);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
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
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const int dd = int_dot8(nib, a[t].q);
        acc[t] += a[t].d * (dsc * (float)dd - dmm * (float)a[t].sum);
      }
    }
  } else {  // W_Q8_0
    int wq[8];
    float d;
    q8_0_decode(row, b, wq, d);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) acc[t] += (d * a[t].d) * (float)int_dot8(wq, a[t].q);
    }
  }
}

template <int WT>
__global__ void __launch_bounds__(kThreads, 1) k_gate_up(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RT = p.T * p.K;
  const int NS = p.gu_nstage;
  const int part_len = kWarps * NT * 2;   // K-split partials: at most kWarps items per stage

  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)NS * p.gu_stage_bytes);
  float* part = reinterpret_cast<float*>(bars + NS);
  GroupSmem g = carve_group(reinterpret_cast<uint8_t*>(part + 2 * part_len), p.E, RT);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  group_routes(p.ids, RT, p.E, g);
  const int S = g.misc[0];
  if (tid == 0) {
    long long W = 0;
    for (int s = 0; s < S; ++s) W += (long long)(p.w0 + g.slot_off[s + 1] - g.slot_off[s]) * p.I;
    const long long lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
    int ub, ib, ue, ie;
    pair_at_cost(lo, g.slot_off, S, p.I, p.w0, ub, ib);
    pair_at_cost(hi, g.slot_off, S, p.I, p.w0, ue, ie);
    g.misc[2] = ub; g.misc[3] = ib; g.misc[4] = ue; g.misc[5] = ie;
    g.misc[6] = 0;
    if (blockIdx.x == 0 && g.misc[1]) atomicOr(p.err, kErrBadId);
  }
  __syncthreads();
  const int ub = g.misc[2], ib = g.misc[3], ue = g.misc[4], ie = g.misc[5];

  // Producer: thread 0 keeps NS stages in flight.
  const uint64_t pol = l2_policy_evict_first();
  PairCursor pc{ub, ib};
  int issued = 0;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      int su, si, sn;
      if (!next_gu_stage(pc, ue, ie, p.I, p.ps, su, si, sn)) break;
      issue_gu_stage(p, stages + (size_t)s * p.gu_stage_bytes, &bars[s], g.slot_e[su], si, sn, pol);
      ++issued;
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // k_prep complete: activations and zeroed counters are visible

  const bool float_act = (WT == W_BF16);
  const bool requant = (p.dn_type != W_BF16);
  const int nb = float_act ? p.H / 8 : p.H / 32;   // blocks (8 values for BF16, 32 otherwise)
  const int max_ks = max(1, nb / 32);

  PairCursor cc{ub, ib};
  int s = 0;
  for (;; ++s) {
    int su, si, sn;
    if (!next_gu_stage(cc, ue, ie, p.I, p.ps, su, si, sn)) break;
    const int buf = s % NS;
    const uint8_t* sbuf = stages + (size_t)buf * p.gu_stage_bytes;
    const int e = g.slot_e[su];
    const uint8_t* gsrc = p.gu_bank + ((size_t)e * 2 * p.I + si) * p.rb_gu;
    const uint8_t* usrc = gsrc + (size_t)p.I * p.rb_gu;
    const uint8_t* gbase = sbuf + (gsrc - align16_down(gsrc));
    const uint8_t* ubase = sbuf + p.gu_up_off + (usrc - align16_down(usrc));
    const int roff = g.slot_off[su];
    const int Tu = g.slot_off[su + 1] - roff;
    const int nch = (Tu + NT - 1) / NT;
    const int base_items = sn * nch;
    const int ks_n = max(1, min(kWarps / base_items, max_ks));
    float* pbuf = part + (s & 1) * part_len;
    const float sg = __ldg(p.scales + 4 * e + 0), su_ = __ldg(p.scales + 4 * e + 1);

    const bool ok = mbar_wait_bounded(&bars[buf], (uint32_t)((s / NS) & 1), kWaitLimit);
    if (!ok) g.misc[6] = 1;
    if (ok) {
      for (int it = warp; it < base_items * ks_n; it += kWarps) {
        const int ks = it / base_items, rem = it % base_items;
        const int pi = rem % sn, ch = rem / sn;
        const int nt = min(NT, Tu - ch * NT);
        int tok[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) tok[t] = (t < nt) ? (int)g.routes[roff + ch * NT + t] / p.K : 0;
        const int b0 = nb * ks / ks_n, b1 = nb * (ks + 1) / ks_n;
        const uint8_t* grow = gbase + (size_t)pi * p.rb_gu;
        const uint8_t* urow = ubase + (size_t)pi * p.rb_gu;
        float accg[NT], accu[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) accg[t] = accu[t] = 0.f;
        if constexpr (WT == W_BF16) {
          for (int c = b0 + lane; c < b1; c += 32) {
            float wg[8], wu[8];
            bf16x8_to_f32(lds128(grow + 16 * c), wg);
            bf16x8_to_f32(lds128(urow + 16 * c), wu);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < nt) {
                float xv[8];
                bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.x + (size_t)tok[t] * p.H + 8 * c)), xv);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  accg[t] = fmaf(wg[j], xv[j], accg[t]);
                  accu[t] = fmaf(wu[j], xv[j], accu[t]);
                }
              }
            }
          }
        } else {
          const int nbh = p.H / 32;
          for (int b = b0 + lane; b < b1; b += 32) {
            ActQ8 a[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t)
              if (t < nt) a[t] = load_act_q8(p.xq, p.xd, p.xsum, (size_t)tok[t] * p.H, (size_t)tok[t] * nbh, b);
            accum_q_block<WT>(grow, p.H, b, a, nt, accg);
            accum_q_block<WT>(urow, p.H, b, a, nt, accu);
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            accg[t] += __shfl_xor_sync(0xffffffffu, accg[t], o);
            accu[t] += __shfl_xor_sync(0xffffffffu, accu[t], o);
          }
        }
        if (lane == 0) {
          if (ks_n == 1) {
            // whole rows in this item: scales, SiLU-GLU and the store happen here
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < nt) {
                const float gv = accg[t] * sg, uv = accu[t] * su_;
                const int r = g.routes[roff + ch * NT + t];
                p.inter[(size_t)r * p.I + si + pi] = __fdiv_rn(gv, 1.0f + expf(-gv)) * uv;
              }
            }
          } else {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              pbuf[(it * NT + t) * 2 + 0] = accg[t];
              pbuf[(it * NT + t) * 2 + 1] = accu[t];
            }
          }
        }
      }
    }
    __syncthreads();
    if (g.misc[6]) break;
    if (tid == 0) {
      int nu, ni, nn;
      if (next_gu_stage(pc, ue, ie, p.I, p.ps, nu, ni, nn)) {
        fence_proxy_async_smem();
        issue_gu_stage(p, stages + (size_t)buf * p.gu_stage_bytes, &bars[buf], g.slot_e[nu], ni, nn, pol);
        ++issued;
      }
    }
    // Epilogue of a K-split stage: fixed-order sum of the partials, scales, SiLU-GLU.
    if (ks_n == 1) continue;
    for (int idx = tid; idx < Tu * sn; idx += kThreads) {
      const int pi = idx % sn, ri = idx / sn;
      const int ch = ri / NT, t = ri % NT;
      float hg = 0.f, hu = 0.f;
      for (int ks = 0; ks < ks_n; ++ks) {
        const int it = ks * base_items + ch * sn + pi;
        hg += pbuf[(it * NT + t) * 2 + 0];
        hu += pbuf[(it * NT + t) * 2 + 1];
      }
      const float gv = hg * sg, uv = hu * su_;
      const float a = __fdiv_rn(gv, 1.0f + expf(-gv)) * uv;
      const int r = g.routes[roff + ri];
      p.inter[(size_t)r * p.I + si + pi] = a;
    }
  }

  if (g.misc[6]) {  // a TMA wait timed out: drain what is in flight (bounded), flag, leave
    if (tid == 0) {
      for (int q = s; q < issued; ++q) mbar_wait_bounded(&bars[q % NS], (uint32_t)((q / NS) & 1), kWaitLimit);
      atomicOr(p.err, kErrTimeout);
    }
    return;
  }
  if (!requant) return;

  // prep_inter: q8_1 requantization of each completed 32-block of the
  // intermediate.  Each CTA adds the pairs it wrote to the block's counter;
  // the CTA that completes a block (counter reaches 32) quantizes it for
  // every route of that expert.
  __syncthreads();
  const int nbi = p.I / 32;
  int j = 0;
  for (int u = ub; u <= ue && u < S; ++u) {
    const int a0 = (u == ub) ? ib : 0;
    const int a1 = (u == ue) ? ie : p.I;
    if (a1 <= a0) continue;
    for (int blk = a0 / 32; blk <= (a1 - 1) / 32; ++blk, ++j) {
      if ((j % kWarps) != warp) continue;
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
      for (int ri = 0; ri < Tu; ++ri) {
        const int r = g.routes[roff + ri];
        const size_t off = (size_t)r * p.I + 32 * (size_t)blk + lane;
        const float v = __ldcg(p.inter + off);
        int q, sum;
        float d;
        q8_1_quantize_warp(v, q, d, sum);
        p.iq[off] = (int8_t)q;
        if (lane == 0) {
          const size_t bi = (size_t)r * nbi + blk;
          p.id[bi] = f16_bits_to_f32(f32_to_f16_bits_rn(d));
          p.isum[bi] = sum;
          p.ish[bi] = (uint16_t)f32_to_f16_bits_rn(d * (float)sum);
        }
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

template <int WT, int LPR>
__global__ void __launch_bounds__(kThreads, 1) k_down(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RT = p.T * p.K;
  const int NS = p.dn_nstage;
  constexpr int RPI = 32 / LPR;   // rows per work item (one per lane group)

  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)NS * p.dn_stage_bytes);
  float* ysm = reinterpret_cast<float*>(bars + NS);
  GroupSmem g = carve_group(reinterpret_cast<uint8_t*>(ysm + (size_t)RT * p.dn_rows_max), p.E, RT);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  group_routes(p.ids, RT, p.E, g);
  const int S = g.misc[0];
  const int j0 = (int)((long long)p.H * blockIdx.x / gridDim.x);
  const int j1 = (int)((long long)p.H * (blockIdx.x + 1) / gridDim.x);
  const int nj = j1 - j0;
  const int sps = p.dn_slots_per_stage, rs = p.dn_rs;
  const int nst = (S > 0 && nj > 0) ? ((nj + rs - 1) / rs) * ((S + sps - 1) / sps) : 0;
  if (tid == 0) g.misc[6] = 0;

  const uint64_t pol = l2_policy_evict_first();
  int issued = 0;
  if (tid == 0) {
    for (; issued < NS && issued < nst; ++issued)
      issue_dn_stage(p, stages + (size_t)issued * p.dn_stage_bytes, &bars[issued], g,
                     down_stage(issued, S, nj, rs, sps), j0, pol);
  }
  pdl_launch_dependents();
  pdl_wait();  // k_gate_up complete: the intermediate is visible
  __syncthreads();

  const int nbi = p.I / 32;
  int k = 0;
  for (; k < nst; ++k) {
    const int buf = k % NS;
    const uint8_t* sbuf = stages + (size_t)buf * p.dn_stage_bytes;
    const DownStage st = down_stage(k, S, nj, rs, sps);
    const bool ok = mbar_wait_bounded(&bars[buf], (uint32_t)((k / NS) & 1), kWaitLimit);
    if (!ok) g.misc[6] = 1;
    if (ok) {
      // items: for each slot of the stage, (row quad, route chunk)
      const int nq = (st.nr + RPI - 1) / RPI;
      int total = 0;
      for (int i = 0; i < st.ns; ++i) {
        const int Tu = g.slot_off[st.u0 + i + 1] - g.slot_off[st.u0 + i];
        total += nq * ((Tu + NT - 1) / NT);
      }
      for (int it = warp; it < total; it += kWarps) {
        int i = 0, rem = it;
        int Tu = 0, nch = 0;
        for (;; ++i) {
          Tu = g.slot_off[st.u0 + i + 1] - g.slot_off[st.u0 + i];
          nch = (Tu + NT - 1) / NT;
          if (rem < nq * nch) break;
          rem -= nq * nch;
        }
        const int u = st.u0 + i;
        const int q = rem % nq, ch = rem / nq;
        const int nt = min(NT, Tu - ch * NT);
        const int grp = lane / LPR, sl = lane % LPR;
        const int row = q * RPI + grp;
        const bool vrow = row < st.nr;
        const int e = g.slot_e[u];
        const uint8_t* src = p.dn_bank + ((size_t)e * p.H + j0 + st.js) * p.rb_dn;
        const uint8_t* rowp = sbuf + (size_t)i * p.dn_piece_bytes + (src - align16_down(src)) +
                              (size_t)(vrow ? row : 0) * p.rb_dn;
        int rt[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) rt[t] = (t < nt) ? (int)g.routes[g.slot_off[u] + ch * NT + t] : 0;
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.f;
        if (vrow) {
          if constexpr (WT == W_BF16) {
            for (int c = sl; c < p.I / 8; c += LPR) {
              float wv[8];
              bf16x8_to_f32(lds128(rowp + 16 * c), wv);
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                if (t < nt) {
                  const float4* ip = reinterpret_cast<const float4*>(p.inter + (size_t)rt[t] * p.I + 8 * c);
                  const float4 v0 = __ldg(ip), v1 = __ldg(ip + 1);
                  acc[t] = fmaf(wv[0], v0.x, acc[t]); acc[t] = fmaf(wv[1], v0.y, acc[t]);
                  acc[t] = fmaf(wv[2], v0.z, acc[t]); acc[t] = fmaf(wv[3], v0.w, acc[t]);
                  acc[t] = fmaf(wv[4], v1.x, acc[t]); acc[t] = fmaf(wv[5], v1.y, acc[t]);
                  acc[t] = fmaf(wv[6], v1.z, acc[t]); acc[t] = fmaf(wv[7], v1.w, acc[t]);
                }
              }
            }
          } else {
            for (int b = sl; b < nbi; b += LPR) {
              ActQ8 a[NT];
#pragma unroll
              for (int t = 0; t < NT; ++t)
                if (t < nt) a[t] = load_act_q8(p.iq, p.id, p.isum, (size_t)rt[t] * p.I, (size_t)rt[t] * nbi, b);
              accum_q_block<WT>(rowp, p.I, b, a, nt, acc);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
        }
        if (sl == 0 && vrow) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < nt) ysm[(size_t)rt[t] * p.dn_rows_max + st.js + row] = acc[t];
        }
      }
    }
    __syncthreads();
    if (g.misc[6]) break;
    if (tid == 0 && issued < nst) {
      fence_proxy_async_smem();
      issue_dn_stage(p, stages + (size_t)buf * p.dn_stage_bytes, &bars[buf], g, down_stage(issued, S, nj, rs, sps),
                     j0, pol);
      ++issued;
    }
  }
  if (g.misc[6]) {
    if (tid == 0) {
      for (int q = k; q < issued; ++q) mbar_wait_bounded(&bars[q % NS], (uint32_t)((q / NS) & 1), kWaitLimit);
      atomicOr(p.err, kErrTimeout);
    }
    return;
  }
  __syncthreads();
  // Route sum in route order k = 0..K-1, then one rounding to bf16.
  for (int idx = tid; idx < p.T * nj; idx += kThreads) {
    const int t = idx / nj, jj = idx % nj;
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
  return (size_t)p.gu_nstage * p.gu_stage_bytes + 8 * (size_t)p.gu_nstage +
         sizeof(float) * 2 * (size_t)kWarps * NT * 2 + group_smem_bytes(p.E, RT);
}

size_t down_smem_bytes(const DecodeParams& p) {
  const int RT = p.T * p.K;
  return (size_t)p.dn_nstage * p.dn_stage_bytes + 8 * (size_t)p.dn_nstage +
         sizeof(float) * (size_t)RT * p.dn_rows_max + group_smem_bytes(p.E, RT);
}

template <typename K>
static cudaError_t launch_pdl(K kernel, int grid, size_t smem, cudaStream_t stream, const DecodeParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
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
  const int work = quantize_x ? (p.T * (p.H / 32) + kWarps - 1) / kWarps : 1;
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

cudaError_t launch_gate_up(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = gate_up_smem_bytes(p);
  cudaError_t e;
  switch (p.gu_type) {
    case W_NVFP4: if ((e = set_smem(k_gate_up<W_NVFP4>, smem))) return e;
      return launch_pdl(k_gate_up<W_NVFP4>, p.g_gu, smem, stream, p);
    case W_Q4_K: if ((e = set_smem(k_gate_up<W_Q4_K>, smem))) return e;
      return launch_pdl(k_gate_up<W_Q4_K>, p.g_gu, smem, stream, p);
    case W_Q8_0: if ((e = set_smem(k_gate_up<W_Q8_0>, smem))) return e;
      return launch_pdl(k_gate_up<W_Q8_0>, p.g_gu, smem, stream, p);
    default: if ((e = set_smem(k_gate_up<W_BF16>, smem))) return e;
      return launch_pdl(k_gate_up<W_BF16>, p.g_gu, smem, stream, p);
  }
}

cudaError_t launch_down(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = down_smem_bytes(p);
  cudaError_t e;
  switch (p.dn_type) {
    case W_NVFP4: if ((e = set_smem(k_down<W_NVFP4, 8>, smem))) return e;
      return launch_pdl(k_down<W_NVFP4, 8>, p.g_dn, smem, stream, p);
    case W_Q4_K: if ((e = set_smem(k_down<W_Q4_K, 8>, smem))) return e;
      return launch_pdl(k_down<W_Q4_K, 8>, p.g_dn, smem, stream, p);
    case W_Q8_0: if ((e = set_smem(k_down<W_Q8_0, 8>, smem))) return e;
      return launch_pdl(k_down<W_Q8_0, 8>, p.g_dn, smem, stream, p);
    default: if ((e = set_smem(k_down<W_BF16, 16>, smem))) return e;
      return launch_pdl(k_down<W_BF16, 16>, p.g_dn, smem, stream, p);
  }
}

// ------------------------------------------------------------------ test hooks

__global__ void k_quantize_blocks(const float* x, int64_t nblocks, uint8_t* out) {
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  if (w >= nblocks) return;
  int q, sum;
  float d;
  q8_1_quantize_warp(x[w * 32 + lane], q, d, sum);
  uint8_t* blk = out + 36 * w;
  blk[4 + lane] = (uint8_t)(int8_t)q;
  if (lane == 0) {
    const uint32_t hdr = f32_to_f16_bits_rn(d) | (f32_to_f16_bits_rn(d * (float)sum) << 16);
    *reinterpret_cast<uint32_t*>(blk) = hdr;
  }
}

cudaError_t launch_quantize_q8_1_blocks(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  const int64_t nb = n / 32;
  if (nb == 0) return cudaSuccess;
  const int64_t grid = (nb * 32 + kThreads - 1) / kThreads;
  k_quantize_blocks<<<(unsigned)grid, kThreads, 0, stream>>>(x, nb, out);
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
    nvfp4_decode(row, k, b, pos, neg, s);
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
