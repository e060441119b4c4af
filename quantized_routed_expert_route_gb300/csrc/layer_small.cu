// Fused routed-expert layer for batches of one or two decode tokens.
//
// One kernel per decode pass instead of k_gate_up + k_down: with so few
// tokens each phase has little work per SM, and a kernel boundary, a second
// route grouping and a second weight-fetch latency cost more than the work.
// Every CTA (one per SM, 16 consumer warps + 1 TMA producer warp):
//   1. waits for the previous grid, groups the routes by expert, takes an even
//      share of the (expert, i) gate/up pairs and H/#CTAs output rows (up to
//      32 routes the producer warp does this alone and starts streaming while
//      the consumers quantize x);
//   2. the producer streams that CTA's gate/up rows and then its down rows of
//      every routed expert through one ring of TMA stages, so the down rows
//      are prefetched while gate_up computes;
//   3. consumers quantize x to q8_1 in shared memory (prep_input), dot every
//      gate and up row with it, apply s_gate / s_up and SiLU-GLU in fp32 and
//      write the fp32 intermediate (FreeToken PR #732, "Design"; Strata PR
//      #292, "Summary/Pipeline");
//   4. a grid barrier (one arrival count per launch, release adds and
//      acquire polls, bounded) makes every CTA's intermediate visible;
//   5. each CTA requantizes the whole intermediate to q8_1 in shared memory
//      (prep_inter), dots its down rows with every route, and sums the routes
//      of a token in route order with w * s_down, writing bf16 with no atomics
//      (FreeToken PR #704, "How it plugs into the CPU executor").
// All CTAs must be resident at once; the launcher checks that one CTA fits on
// every SM and uses this kernel only then.
#include "decode_common.cuh"

namespace qre {

constexpr int kLsWarps = 16;
constexpr int kLsConsumers = 32 * kLsWarps;
constexpr int kLsThreads = kLsConsumers + 32;
constexpr unsigned kGridSpinLimit = 1u << 21;   // polling rounds of the barrier words (~2 s) before giving up

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier over all CTAs of the grid.  bar[0] is an epoch that only changes
// between launches; the launch of epoch n counts its arrivals in the word
// bar[32 * (1 + n % 2)] (its own 128-byte line), which the previous launch
// left at zero.  Arriving, thread 0 of a CTA adds 1 with release semantics
// (publishing the CTA's earlier writes, ordered before it by the consumer
// barrier) and polls the count with acquire loads until every CTA has
// arrived.  After the barrier CTA 0 zeroes the other count (the next
// launch's) and advances the epoch (every CTA read it before arriving, so
// before CTA 0 could pass).  The wait is bounded: on timeout the error word
// is flagged and the CTA goes on (its results are then invalid, but nothing
// hangs; the launch after next starts from a zeroed count again).
__device__ void ls_grid_barrier(unsigned* bar, unsigned epoch, uint32_t* err) {
  consumer_sync<kLsConsumers>();
  if (threadIdx.x == 0) {
    unsigned* cnt = bar + 32 * (1 + (epoch & 1u));
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
    unsigned spins = 0;
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= gridDim.x) break;
      if (++spins > kGridSpinLimit) {
        atomicOr(err, kErrTimeout);
        break;
      }
    }
    if (blockIdx.x == 0) {
      st_relaxed_gpu(bar + 32 * (1 + ((epoch + 1u) & 1u)), 0u);
      st_relaxed_gpu(bar, epoch + 1u);
    }
  }
  consumer_sync<kLsConsumers>();
}

// q8_1 quantization of `nblk` 32-value blocks (bf16 or fp32 values, row-major)
// into shared-memory planes, one lane quad per block.  Blocks of rows whose
// route is invalid (rvalid[row] == 0) are skipped.  CTA 0 mirrors the blocks
// to the workspace planes for inspection.
template <bool kBf16In>
__device__ void ls_quantize(const void* src, int nblk, const uint8_t* rvalid, int blocks_per_row, int8_t* q, float* d,
                            int* sm, bool mirror, int8_t* wq, float* wd, int* wsum, uint16_t* wsh) {
  const int quad = threadIdx.x >> 2, ql = threadIdx.x & 3;
  constexpr int kQuads = kLsConsumers / 4;
  constexpr int kR = 4;   // blocks per quad per round, all loads issued first
  for (int b0 = 0; b0 < nblk; b0 += kR * kQuads) {
    float v[kR][8];
    bool on[kR];
#pragma unroll
    for (int h = 0; h < kR; ++h) {
      const int b = b0 + h * kQuads + quad;
      on[h] = b < nblk && (!rvalid || rvalid[b / blocks_per_row]);
      if (on[h]) {
        const size_t off = (size_t)b * 32 + 8 * ql;
        if constexpr (kBf16In) {
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + off)), v[h]);
        } else {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + off);
          const float4 a = __ldcg(p), c = __ldcg(p + 1);
          v[h][0] = a.x; v[h][1] = a.y; v[h][2] = a.z; v[h][3] = a.w;
          v[h][4] = c.x; v[h][5] = c.y; v[h][6] = c.z; v[h][7] = c.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[h][i] = 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < kR; ++h) {
      if (b0 + h * kQuads + 8 * (int)(threadIdx.x >> 5) >= nblk) break;   // none of this warp's quads has a block
      uint32_t w0, w1;
      float dd;
      int sum;
      q8_1_quantize_quad(v[h], w0, w1, dd, sum);
      if (on[h]) {
        const int b = b0 + h * kQuads + quad;
        const size_t off = (size_t)b * 32 + 8 * ql;
        *reinterpret_cast<uint2*>(q + off) = make_uint2(w0, w1);
        const float dh = f16_bits_to_f32(f32_to_f16_bits_rn(dd));
        if (ql == 0) {
          d[b] = dh;
          sm[b] = sum;
        }
        if (mirror) {
          *reinterpret_cast<uint2*>(wq + off) = make_uint2(w0, w1);
          if (ql == 0) {
            wd[b] = dh;
            wsum[b] = sum;
            wsh[b] = (uint16_t)f32_to_f16_bits_rn(dd * (float)sum);
          }
        }
      }
    }
  }
}

template <int WG, int WD, int LPR>
__global__ void __launch_bounds__(kLsThreads, 1) k_layer_small(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RT = p.T * p.K;
  const int NS = p.ls_ns;
  const int SB = p.ls_sb;
  constexpr int RPI = 32 / LPR;

  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * SB);
  uint64_t* empty = full + NS;
  uint64_t* grouped = empty + NS;   // small batches: the producer warp's grouping and split are published
  uint8_t* xact = reinterpret_cast<uint8_t*>(grouped + 1);
  xact += (16 - (reinterpret_cast<uintptr_t>(xact) & 15)) & 15;
  uint8_t* iact = xact + p.gu_act_bytes;
  float* ysm = reinterpret_cast<float*>(iact + p.dn_act_bytes);
  float* swd = ysm + (size_t)RT * p.dn_rows_max;                       // [RT] s_down * w (0: bad route)
  uint8_t* rvalid = reinterpret_cast<uint8_t*>(swd + RT);
  uint8_t* gbase_smem = rvalid + RT;
  gbase_smem += (16 - (reinterpret_cast<uintptr_t>(gbase_smem) & 15)) & 15;
  GroupSmem g = carve_group(gbase_smem, p.E, RT);

  // Up to 32 routes the producer warp groups the routes and splits the
  // pairs itself and starts streaming at once, while the consumers quantize
  // x; they meet at the `grouped` barrier.  More routes: the whole CTA groups.
  const bool small = RT <= 32;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLsWarps);
    }
    mbar_init(grouped, 1);
    fence_mbar_init();
  }
  if (small && warp == kLsWarps) {
    // the lines of ids, weights and x into L2 while the previous grid finishes
    // (prefetches only: every load of them comes after griddepcontrol.wait)
    if (lane == 0) prefetch_l2(p.ids);
    if (lane == 1) prefetch_l2(p.w);
    for (int i = lane; i < (2 * p.T * p.H + 127) / 128; i += 32) prefetch_l2(reinterpret_cast<const uint8_t*>(p.x) + 128 * i);
  }
  __syncthreads();   // the mbarriers are initialised
  pdl_wait();   // x and ids may come from the previous grid
  pdl_launch_dependents();
  // the barrier epoch (written by the previous launch); a relaxed load, so
  // it does not hold up this thread's later work
  const unsigned epoch = (tid == 0) ? ld_relaxed_gpu(p.bar) : 0u;
  if (!small) group_routes(p.ids, RT, p.E, p.K, g);
  else if (warp == kLsWarps) group_routes_small_warp(p.ids, RT, p.E, p.K, g, lane);
  if (small && warp == kLsWarps) {
    __syncwarp();
    const int S = g.misc[0];
    // every expert has about one route, so split the pairs evenly (32-bit
    // arithmetic when the products fit)
    if (lane == 0) {
    const unsigned P = (unsigned)S * (unsigned)p.I;
    unsigned lo, hi;
    if (P <= 0xFFFFFFFFu / gridDim.x) {
      lo = P * blockIdx.x / gridDim.x;
      hi = P * (blockIdx.x + 1) / gridDim.x;
    } else {
      lo = (unsigned)((unsigned long long)P * blockIdx.x / gridDim.x);
      hi = (unsigned)((unsigned long long)P * (blockIdx.x + 1) / gridDim.x);
    }
    g.misc[2] = lo / p.I;
    g.misc[3] = lo - (lo / p.I) * p.I;
    g.misc[4] = hi / p.I;
    g.misc[5] = hi - (hi / p.I) * p.I;
    g.misc[6] = 0;
    g.misc[7] = 0;
    if (blockIdx.x == 0 && g.misc[1]) atomicOr(p.err, kErrBadId);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(grouped);   // after the warp's grouping and the split (release)
  } else if (!small && warp == 0) {
    const int S = g.misc[0];
    // Split of the S*I (gate, up) pairs, balanced by cost: a pair costs its
    // row bytes plus one decode-and-dot per route of its expert, so cost =
    // 1 + routes of the slot.
    long long W = 0;
    for (int sl = lane; sl < S; sl += 32) W += 1 + g.slot_off[sl + 1] - g.slot_off[sl];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    W *= p.I;
    int ub, ib, ue, ie;
    pair_at_cost_warp(cost_cut(W, blockIdx.x, gridDim.x), g.slot_off, S, p.I, 1, lane, ub, ib);
    pair_at_cost_warp(cost_cut(W, blockIdx.x + 1, gridDim.x), g.slot_off, S, p.I, 1, lane, ue, ie);
    if (lane == 0) {
      g.misc[2] = ub;
      g.misc[3] = ib;
      g.misc[4] = ue;
      g.misc[5] = ie;
      g.misc[6] = 0;
      g.misc[7] = 0;
      if (blockIdx.x == 0 && g.misc[1]) atomicOr(p.err, kErrBadId);
    }
  }
  if (!small) __syncthreads();
  const int j0 = (int)((unsigned)p.H * blockIdx.x / gridDim.x);
  const int j1 = (int)((unsigned)p.H * (blockIdx.x + 1) / gridDim.x);
  const int nj = j1 - j0;
  const int sps = p.dn_slots_per_stage, rs = p.dn_rs;

  if (warp == kLsWarps) {
    // TMA producer: this CTA's gate/up stages, then its down stages, through one ring.
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int ub = g.misc[2], ib = g.misc[3], ue = g.misc[4], ie = g.misc[5];
      PairCursor pc{ub, ib};
      int buf = 0;
      uint32_t eph = 0;
      bool wrapped = false, ok = true;
      int k = 0, nst_dn = -1;
      for (;;) {
        int su = 0, si = 0, sn = 0;
        const bool gu = next_gu_stage(pc, ue, ie, p.I, p.ps, su, si, sn);
        if (!gu && nst_dn < 0) {   // the down stage count, once the gate/up stages are out
          const int S = g.misc[0];
          nst_dn = (S > 0 && nj > 0) ? ((nj + rs - 1) / rs) * ((S + sps - 1) / sps) : 0;
        }
        if (!gu && k >= nst_dn) break;
        if (wrapped) {
          if (!mbar_wait_bounded(&empty[buf], eph, kWaitLimit)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
        }
        uint8_t* dst = ring + (size_t)buf * SB;
        if (gu) issue_gu_stage(p, dst, &full[buf], g.slot_e[su], si, sn, pol);
        else issue_dn_stage(p, dst, &full[buf], g, down_stage(k++, g.misc[0], nj, rs, sps), j0, pol);
        atomicAdd(&g.misc[7], 1);
        if (++buf == NS) {
          buf = 0;
          if (wrapped) eph ^= 1u;
          wrapped = true;
        }
      }
      if (!ok) g.misc[6] = 1;
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp;
  const int nbh = p.H / 32, nbi = p.I / 32;
  int8_t* xq = reinterpret_cast<int8_t*>(xact);
  float* xd = reinterpret_cast<float*>(xact + (size_t)p.T * p.H);
  int* xs = reinterpret_cast<int*>(xd + (size_t)p.T * nbh);
  if (small) {
    // x first (it needs no grouping), then the producer's grouping and split
    if constexpr (is_float_w(WG)) {
      copy_to_smem<kLsConsumers>(xact, p.x, 2 * (size_t)p.T * p.H);
    } else {
      ls_quantize<true>(p.x, p.T * nbh, nullptr, nbh, xq, xd, xs, blockIdx.x == 0, p.xq, p.xd, p.xsum, p.xsh);
    }
    if (!mbar_wait_bounded(grouped, 0u, kWaitLimit)) {
      if (tid == 0) atomicOr(p.err, kErrTimeout);
      return;
    }
  }
  const int S = g.misc[0];
  const int ub = g.misc[2], ib = g.misc[3], ue = g.misc[4], ie = g.misc[5];
  const int ngrp = (S + sps - 1) / sps;
  const int nst_dn = (S > 0 && nj > 0) ? ((nj + rs - 1) / rs) * ngrp : 0;
  // route validity and s_down * w of every route, from the grouping (off the
  // producer's path: the producer is already streaming)
  for (int r = tid; r < RT; r += kLsConsumers) {
    rvalid[r] = 0;
    swd[r] = 0.f;
  }
  consumer_sync<kLsConsumers>();
  for (int sl = tid; sl < S; sl += kLsConsumers) {
    const int e = g.slot_e[sl];
    const float sd = __ldg(p.scales + 4 * e + 2);
    for (int i = g.slot_off[sl]; i < g.slot_off[sl + 1]; ++i) {
      const int r = g.routes[i];
      rvalid[r] = 1;
      swd[r] = sd * __ldg(p.w + r);
    }
  }
  for (int sl = tid; sl < S; sl += kLsConsumers) {
    const int e = g.slot_e[sl];
    g.sscale[3 * sl + 0] = __ldg(p.scales + 4 * e + 0);
    g.sscale[3 * sl + 1] = __ldg(p.scales + 4 * e + 1);
  }
  if (!small) {
    if constexpr (is_float_w(WG)) {
      copy_to_smem<kLsConsumers>(xact, p.x, 2 * (size_t)p.T * p.H);
    } else {
      ls_quantize<true>(p.x, p.T * nbh, nullptr, nbh, xq, xd, xs, blockIdx.x == 0, p.xq, p.xd, p.xsum, p.xsh);
    }
  }
  consumer_sync<kLsConsumers>();

  // gate_up: pairs round-robin over the warps, routes of the expert inside
  const size_t rbg = (size_t)p.rb_gu;
  PairCursor cc{ub, ib};
  int rot = 0, buf = 0, consumed = 0;
  uint32_t fph = 0;
  for (;;) {
    int su, si, sn;
    if (!next_gu_stage(cc, ue, ie, p.I, p.ps, su, si, sn)) break;
    const uint8_t* sbuf = ring + (size_t)buf * SB;
    const int e = g.slot_e[su];
    const uint8_t* gsrc = p.gu_bank + ((size_t)e * 2 * p.I + si) * rbg;
    const uint8_t* usrc = gsrc + (size_t)p.I * rbg;
    const uint8_t* gbase = sbuf + (gsrc - align16_down(gsrc));
    const uint8_t* ubase = sbuf + p.gu_up_off + (usrc - align16_down(usrc));
    const int roff = g.slot_off[su];
    const int Tu = g.slot_off[su + 1] - roff;
    const float sg = g.sscale[3 * su + 0], su_ = g.sscale[3 * su + 1];
    if (!mbar_wait_bounded(&full[buf], fph, kWaitLimit)) {
      g.misc[6] = 1;
      break;
    }
    for (int pi = (cw - rot) & (kLsWarps - 1); pi < sn; pi += kLsWarps) {
      const uint8_t* grow = gbase + (size_t)pi * rbg;
      const uint8_t* urow = ubase + (size_t)pi * rbg;
      for (int ri = 0; ri < Tu; ++ri) {
        const int t = g.rtok[roff + ri];
        float2 h;
        if constexpr (is_float_w(WG)) {
          ActSrc act;
          act.xb = reinterpret_cast<const uint16_t*>(xact);
          act.n = p.H;
          int tok[NT] = {t, 0, 0, 0};
          float ag[NT], au[NT];
          gu_item<WG, 1>(grow, urow, p.H, 0, p.H / 8, lane, act, tok, 1, ag, au);
          h = make_float2(ag[0], au[0]);
        } else {
          h = gu_pair_q8<WG>(grow, urow, p.H, lane, xq + (size_t)t * p.H, xd + t * nbh, xs + t * nbh);
        }
        if (lane == 0) {
          const int r = g.routes[roff + ri];
          p.inter[(size_t)r * p.I + si + pi] = glu_act(h.x * sg, h.y * su_, p.glu);
        }
      }
    }
    rot = (rot + sn) & (kLsWarps - 1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[buf]);
    ++consumed;
    if (++buf == NS) {
      buf = 0;
      fph ^= 1u;
    }
  }

  // every CTA's intermediate is written before any CTA reads it
  ls_grid_barrier(p.bar, epoch, p.err);

  // prep_inter
  int8_t* iq = reinterpret_cast<int8_t*>(iact);
  float* idd = reinterpret_cast<float*>(iact + (size_t)RT * p.I);
  int* is = reinterpret_cast<int*>(idd + (size_t)RT * nbi);
  ActSrc dact;
  dact.n = p.I;
  dact.xf = p.inter;
  if constexpr (is_float_w(WD)) {
    if (p.dn_act_smem) {
      copy_to_smem<kLsConsumers>(iact, p.inter, 4 * (size_t)RT * p.I);
      dact.xf = reinterpret_cast<const float*>(iact);
    }
  } else {
    ls_quantize<false>(p.inter, RT * nbi, rvalid, nbi, iq, idd, is, blockIdx.x == 0, p.iq, p.id, p.isum, p.ish);
  }
  consumer_sync<kLsConsumers>();

  // down: (slot, row group) items round-robin over the warps, routes inside
  const size_t rbd = (size_t)p.rb_dn;
  const int grp = lane / LPR, sl = lane % LPR;
  rot = 0;
  int k = 0;
  for (; k < nst_dn && !g.misc[6]; ++k) {
    const uint8_t* sbuf = ring + (size_t)buf * SB;
    const DownStage st = down_stage(k, S, nj, rs, sps);
    const int nq = (st.nr + RPI - 1) / RPI;
    if (!mbar_wait_bounded(&full[buf], fph, kWaitLimit)) {
      g.misc[6] = 1;
      break;
    }
    for (int i = 0; i < st.ns; ++i) {
      const int u = st.u0 + i;
      const int roff = g.slot_off[u];
      const int Tu = g.slot_off[u + 1] - roff;
      const int e = g.slot_e[u];
      const uint8_t* src = p.dn_bank + ((size_t)e * p.H + j0 + st.js) * rbd;
      const uint8_t* piece = sbuf + (size_t)i * p.dn_piece_bytes + (src - align16_down(src));
      for (int q = (cw - rot) & (kLsWarps - 1); q < nq; q += kLsWarps) {
        const int row = q * RPI + grp;
        const bool vrow = row < st.nr;
        const uint8_t* rowp = piece + (size_t)(vrow ? row : 0) * rbd;
        for (int ri = 0; ri < Tu; ++ri) {
          const int r = g.routes[roff + ri];
          float v;
          if constexpr (is_float_w(WD)) {
            int rt[NT] = {r, 0, 0, 0};
            float res[NT];
            dn_item<WD, LPR, 1>(rowp, vrow, p.I, sl, dact, rt, 1, res);
            v = res[0];
          } else {
            v = dn_row_q8<WD, LPR>(rowp, vrow, p.I, sl, iq + (size_t)r * p.I, idd + r * nbi, is + r * nbi);
          }
          if (vrow && sl == 0) ysm[(size_t)r * p.dn_rows_max + st.js + row] = v;
        }
      }
      rot = (rot + nq) & (kLsWarps - 1);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[buf]);
    ++consumed;
    if (++buf == NS) {
      buf = 0;
      fph ^= 1u;
    }
  }
  consumer_sync<kLsConsumers>();
  if (g.misc[6]) {  // a bounded wait ran out: drain what is in flight (bounded), flag, leave
    if (tid == 0) {
      const int issued = g.misc[7];
      for (int qn = consumed; qn < issued; ++qn)
        mbar_wait_bounded(&full[qn % NS], (uint32_t)((qn / NS) & 1), kWaitLimit);
      atomicOr(p.err, kErrTimeout);
    }
    return;
  }
  // route sum in route order k = 0..K-1, then one rounding to bf16
  for (int idx = tid; idx < p.T * nj; idx += kLsConsumers) {
    const int t = idx / nj, jj = idx - t * nj;
    float acc = 0.f;
    for (int kk = 0; kk < p.K; ++kk) {
      const int r = t * p.K + kk;
      if (!rvalid[r]) continue;
      acc += ysm[(size_t)r * p.dn_rows_max + jj] * swd[r];
    }
    p.out[(size_t)t * p.H + j0 + jj] = (uint16_t)f32_to_bf16_bits_rn(acc);
  }
}

// ------------------------------------------------------------------ launch

size_t layer_small_smem_bytes(const DecodeParams& p) {
  const int RT = p.T * p.K;
  return (size_t)p.ls_ns * p.ls_sb + 16 * (size_t)p.ls_ns + 32 + (size_t)p.gu_act_bytes + (size_t)p.dn_act_bytes +
         sizeof(float) * (size_t)RT * (p.dn_rows_max + 1) + (size_t)RT + 16 + group_smem_bytes(p.E, RT);
}

template <int WG, int WD, int LPR>
static cudaError_t launch_ls_t(const DecodeParams& p, cudaStream_t stream, bool probe_only, bool* fits) {
  const size_t smem = layer_small_smem_bytes(p);
  cudaError_t e = cudaFuncSetAttribute(k_layer_small<WG, WD, LPR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (fits) *fits = false;
    return probe_only ? cudaSuccess : e;
  }
  if (probe_only) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_layer_small<WG, WD, LPR>, kLsThreads, smem);
    if (fits) *fits = (e == cudaSuccess && per_sm >= 1);
    cudaGetLastError();
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.g_ls);
  cfg.blockDim = dim3(kLsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // Cooperative: the driver keeps every CTA resident at once, which the grid
  // barrier needs; programmatic serialization: the next layer's grid may be
  // scheduled early (it waits before touching anything this one writes).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_layer_small<WG, WD, LPR>, p);
}

// Same-type layers of every format (aligned NVFP4 rows) and the Q4_K gate_up
// + Q6_K down pair of Q4_K_M checkpoints; other pairs use the two-kernel path.
static cudaError_t dispatch_ls(const DecodeParams& p, cudaStream_t stream, bool probe_only, bool* fits) {
  if (p.gu_type == W_Q4_K && p.dn_type == W_Q6_K) return launch_ls_t<W_Q4_K, W_Q6_K, 4>(p, stream, probe_only, fits);
  if (p.gu_type != p.dn_type) {
    if (fits) *fits = false;
    return cudaSuccess;
  }
  switch (p.gu_type) {
    case W_NVFP4:
      if (p.rb_gu % 16 != 0 || p.rb_dn % 16 != 0) {
        if (fits) *fits = false;
        return cudaSuccess;
      }
      return launch_ls_t<W_NVFP4, W_NVFP4, 4>(p, stream, probe_only, fits);
    case W_Q4_K: return launch_ls_t<W_Q4_K, W_Q4_K, 4>(p, stream, probe_only, fits);
    case W_Q8_0: return launch_ls_t<W_Q8_0, W_Q8_0, 8>(p, stream, probe_only, fits);
    case W_Q6_K: return launch_ls_t<W_Q6_K, W_Q6_K, 4>(p, stream, probe_only, fits);
    case W_Q4_0: return launch_ls_t<W_Q4_0, W_Q4_0, 8>(p, stream, probe_only, fits);
    case W_Q4_1: return launch_ls_t<W_Q4_1, W_Q4_1, 8>(p, stream, probe_only, fits);
    case W_Q5_0: return launch_ls_t<W_Q5_0, W_Q5_0, 8>(p, stream, probe_only, fits);
    case W_Q5_1: return launch_ls_t<W_Q5_1, W_Q5_1, 8>(p, stream, probe_only, fits);
    case W_Q5_K: return launch_ls_t<W_Q5_K, W_Q5_K, 4>(p, stream, probe_only, fits);
    case W_MXFP4: return launch_ls_t<W_MXFP4, W_MXFP4, 8>(p, stream, probe_only, fits);
    case W_F16: return launch_ls_t<W_F16, W_F16, 16>(p, stream, probe_only, fits);
    case W_F32: return launch_ls_t<W_F32, W_F32, 16>(p, stream, probe_only, fits);
    default: return launch_ls_t<W_BF16, W_BF16, 16>(p, stream, probe_only, fits);
  }
}

bool layer_small_fits(const DecodeParams& p) {
  bool fits = false;
  dispatch_ls(p, nullptr, true, &fits);
  return fits;
}

cudaError_t launch_layer_small(const DecodeParams& p, cudaStream_t stream) {
  return dispatch_ls(p, stream, false, nullptr);
}

}  // namespace qre
