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
//
// The kernel templates live in decode_twok.cuh; this file instantiates them
// for BF16, Q8_0, Q4_K and NVFP4 rows, decode_types_b.cu and
// decode_types_c.cu for the other GGUF types.
#include "decode_twok.cuh"

namespace qre {

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

// MAXNT = 1 (batches of up to two tokens): the x quantizer runs inside this
// kernel, which waits for the previous grid before touching ids, and the
// intermediate is requantized by k_down.  MAXNT = 4: k_prep quantizes x and
// has already waited, so ids are read before this kernel waits, and the
// intermediate is requantized here by the last CTA to finish each block.
// Launch bounds keep registers low enough for a k_down CTA to share the SM.

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

cudaError_t launch_prep(const DecodeParams& p, cudaStream_t stream) {
  const int quantize_x = is_float_w(p.gu_type) ? 0 : 1;
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

cudaError_t launch_gate_up(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = gate_up_smem_bytes(p);
  switch (p.gu_type) {
    case W_NVFP4:
      if (p.rb_gu % 16 != 0) return launch_gu_w<W_NVFP4_U>(p, smem, stream);
      return launch_gu_w<W_NVFP4>(p, smem, stream);
    case W_Q4_K: return launch_gu_w<W_Q4_K>(p, smem, stream);
    case W_Q8_0: return launch_gu_w<W_Q8_0>(p, smem, stream);
    case W_Q6_K: case W_Q4_0: case W_Q4_1: return launch_gate_up_types_b(p, smem, stream);
    case W_Q5_0: case W_Q5_1: case W_Q5_K: case W_MXFP4: case W_F16: case W_F32:
      return launch_gate_up_types_c(p, smem, stream);
    default: return launch_gu_w<W_BF16>(p, smem, stream);
  }
}

cudaError_t launch_down(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = down_smem_bytes(p);
  switch (p.dn_type) {
    case W_NVFP4:
      if (p.rb_dn % 16 != 0) return launch_dn_w<W_NVFP4_U, 8>(p, smem, stream);
      return launch_dn_w<W_NVFP4, 8>(p, smem, stream);
    case W_Q4_K: return launch_dn_w<W_Q4_K, 8>(p, smem, stream);
    case W_Q8_0: return launch_dn_w<W_Q8_0, 8>(p, smem, stream);
    case W_Q6_K: case W_Q4_0: case W_Q4_1: return launch_down_types_b(p, smem, stream);
    case W_Q5_0: case W_Q5_1: case W_Q5_K: case W_MXFP4: case W_F16: case W_F32:
      return launch_down_types_c(p, smem, stream);
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
#pragma unroll
  for (int i = 0; i < 8; ++i) a.sum = __dp4a(a.q[i], 0x01010101, a.sum);
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
  } else if (type == W_Q6_K) {
    int wq[8];
    float d, s0, s1;
    q6k_decode(row, b, wq, d, s0, s1);
    int d0, d1;
    int_dots_halves(wq, a.q, d0, d1);
    out[(size_t)r * (k / 16) + 2 * b] = d0;
    out[(size_t)r * (k / 16) + 2 * b + 1] = d1;
  } else if (type == W_Q4_0) {
    int wq[8];
    float d;
    q4_0_decode(row, b, wq, d);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q) - 8 * a.sum;
  } else if (type == W_Q4_1 || type == W_Q5_1) {
    int wq[8];
    float d, m;
    if (type == W_Q4_1) q4_1_decode(row, b, wq, d, m);
    else q5_1_decode(row, b, wq, d, m);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q);
  } else if (type == W_Q5_0) {
    int wq[8];
    float d;
    q5_0_decode(row, b, wq, d);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q) - 16 * a.sum;
  } else if (type == W_Q5_K) {
    int wq[8];
    float dsc, dmm;
    q5k_decode(row, b, wq, dsc, dmm);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q);
  } else if (type == W_MXFP4) {
    int wq[8];
    float sc;
    mxfp4_decode(row, b, wq, sc);
    out[(size_t)r * nb + b] = int_dot8(wq, a.q);
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

// Test hook: one of the kernels' bounded waits on an mbarrier whose phase
// nothing ever completes (it expects one arrival that never comes), with a
// short limit.  mode 0: mbar_wait_bounded, `limit` sleeping polls (the form
// the decode kernels use); mode 1: mbar_wait_spin, `limit` microseconds of
// device time (the grouped and prompt-path kernels).  When the wait runs out
// the kernel ORs kErrTimeout into *err and returns, as those kernels do.
__global__ void k_wait_timeout(int mode, uint32_t limit, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = (mode == 0) ? mbar_wait_bounded(&bar, 0u, limit)
                                : mbar_wait_spin(&bar, 0u, 1000ull * (unsigned long long)limit);
    if (!ok) atomicOr(err, kErrTimeout);
  }
}

cudaError_t launch_wait_timeout(int mode, uint32_t limit, uint32_t* err, cudaStream_t stream) {
  k_wait_timeout<<<1, 32, 0, stream>>>(mode, limit, err);
  return cudaGetLastError();
}

}  // namespace qre
