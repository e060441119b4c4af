// The two-kernel decode path's gate_up and down kernels as templates over
// the row type, and their launchers.  Shared by the translation units that
// instantiate them (decode.cu and decode_types_*.cu), so that the
// instantiations for the many row types compile in parallel.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace qre {

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
  if (is_float_w(WT)) {
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

  const bool requant = !kFused && (!is_float_w(p.dn_type));
  const int nb = (is_float_w(WT)) ? p.H / 8 : p.H / 32;   // blocks (8 values for BF16, 32 otherwise)
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
    if (kFused && !is_float_w(WT) && ks_n == 1) {
      // one or two tokens: activations are shared-memory q8_1 planes; each
      // warp takes whole pairs, routes of the expert one after another
      const int8_t* aqs = reinterpret_cast<const int8_t*>(actm);
      const float* ads = reinterpret_cast<const float*>(actm + (size_t)p.T * p.H);
      const int* ass = reinterpret_cast<const int*>(ads + (size_t)p.T * (p.H >> 5));
      for (int pi = (cw - rot) & (kConsumerWarps - 1); pi < sn; pi += kConsumerWarps) {
        const uint8_t* grow = gbase + (size_t)pi * rbg;
        const uint8_t* urow = ubase + (size_t)pi * rbg;
        for (int ri = 0; ri < Tu; ++ri) {
          const int t = g.rtok[roff + ri];
          const float2 h = gu_pair_q8<WT>(grow, urow, p.H, lane, aqs + (size_t)t * p.H, ads + t * (p.H >> 5),
                                          ass + t * (p.H >> 5));
          if (lane == 0) {
            const int r = g.routes[roff + ri];
            p.inter[(size_t)r * p.I + si + pi] = glu_act(h.x * sg, h.y * su_, p.glu);
          }
        }
      }
      rot = (rot + sn) & (kConsumerWarps - 1);
    } else if (ks_n == 1) {
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
            p.inter[(size_t)r * p.I + si + pi] = glu_act(gv * sg, uv * su_, p.glu);
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
          p.inter[(size_t)r * p.I + si + pi] = glu_act(hg * sg, hu * su_, p.glu);
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
  const int j0 = (int)((unsigned)p.H * blockIdx.x / gridDim.x);
  const int j1 = (int)((unsigned)p.H * (blockIdx.x + 1) / gridDim.x);
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
  if (is_float_w(WT)) {
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
      if constexpr (kFused && !is_float_w(WT)) {
        // one or two tokens: the requantized intermediate is in shared memory
        const int8_t* aqs = reinterpret_cast<const int8_t*>(actm);
        const float* ads = reinterpret_cast<const float*>(actm + (size_t)RT * p.I);
        const int* ass = reinterpret_cast<const int*>(ads + (size_t)RT * (p.I >> 5));
        for (int q = (cw - rot) & (kConsumerWarps - 1); q < nq; q += kConsumerWarps) {
          const int row = q * RPI + grp;
          const bool vrow = row < st.nr;
          const uint8_t* rowp = piece + (size_t)(vrow ? row : 0) * rbd;
          for (int ri = 0; ri < Tu; ++ri) {
            const int r = g.routes[roff + ri];
            const float v = dn_row_q8<WT, LPR>(rowp, vrow, p.I, sl, aqs + (size_t)r * p.I, ads + r * (p.I >> 5),
                                               ass + r * (p.I >> 5));
            if (vrow && sl == 0) ysm[(size_t)r * p.dn_rows_max + st.js + row] = v;
          }
        }
      } else {
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

// Launchers of the row types instantiated outside decode.cu.
cudaError_t launch_gate_up_types_b(const DecodeParams& p, size_t smem, cudaStream_t stream);
cudaError_t launch_down_types_b(const DecodeParams& p, size_t smem, cudaStream_t stream);
cudaError_t launch_gate_up_types_c(const DecodeParams& p, size_t smem, cudaStream_t stream);
cudaError_t launch_down_types_c(const DecodeParams& p, size_t smem, cudaStream_t stream);

}  // namespace qre
