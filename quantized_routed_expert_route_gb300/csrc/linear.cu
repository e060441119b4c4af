// Dense quantized linear with a per-output-row scale in the epilogue:
//
//   out[t, n] = bf16(row_scale[n] * sum_k W[n, k] * q8_1(x[t])[k])
//
// FreeToken PR #732, "Design": a dense linear multiplies its matmul result by
// its scale, and a fused module (qkv, gate_up) carries ggml_scale, one fp32
// value per output row; its "Not covered" list applies that scale in a
// separate elementwise kernel after the GEMM.  Here it is a multiply in the
// epilogue of the one kernel that reads the rows.
//
// A decode-sized batch (T <= 8 tokens) makes this a matrix-vector product
// bound by the bytes of W.  One CTA per SM owns a contiguous range of rows;
// its producer warp streams the range through a ring of shared-memory slots
// with 1-D TMA bulk copies (a slot holds whole rows, copied from the 16-byte
// boundary at or below the first row), while 15 consumer warps quantize x to
// q8_1 once into shared memory and then take the slot's rows one per warp:
// lanes stride the 32-value blocks of a row, each block's exact integer dot
// with every token's q8_1 block is scaled in fp32 (the same block functions
// as the routed-expert path), a warp reduction sums the lanes, and lane t
// writes token t's output.  Every wait is bounded in device time; on a
// timeout the CTA raises the error word and lets its copies in flight land.
#include "decode_common.cuh"

namespace qre {

namespace {

constexpr int kLinConsumerWarps = 15;   // 16 warps in all: 4 per SM sub-partition, up to 128 registers a thread
constexpr int kLinConsumers = 32 * kLinConsumerWarps;
constexpr int kLinThreads = kLinConsumers + 32;           // + one TMA producer warp
constexpr int kLinMaxStages = 8;
constexpr uint64_t kLinWaitNs = 2000000000ull;            // one wait gives up after 2 s of device time

__device__ __forceinline__ bool lin_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kLinWaitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

template <int WT, int LT>
__global__ void __launch_bounds__(kLinThreads, 1) k_linear(const __grid_constant__ LinParams p) {
  extern __shared__ __align__(128) uint8_t lin_smem[];
  __shared__ uint64_t full_bar[kLinMaxStages], empty_bar[kLinMaxStages];
  __shared__ volatile int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int r_begin = (int)((long long)p.N * blockIdx.x / G);
  const int r_end = (int)((long long)p.N * (blockIdx.x + 1) / G);
  const int nst = (r_end - r_begin + p.rps - 1) / p.rps;
  uint8_t* ring = lin_smem + p.act_bytes;
  volatile int* abort = &abort_flag;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kLinConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kLinConsumerWarps) {
    // ---------------- producer: the CTA's rows, slot by slot
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();   // weight rows: read once
      int i = 0;
      bool ok = true;
      for (; i < nst; ++i) {
        const int s = i % p.nstage;
        const uint32_t u = (uint32_t)(i / p.nstage);
        if (u >= 1 && !lin_wait(&empty_bar[s], (u - 1) & 1u, abort)) {
          ok = false;
          break;
        }
        const int r0 = r_begin + i * p.rps;
        const int n = min(p.rps, r_end - r0);
        const uint8_t* src = p.rows + (size_t)r0 * p.rb;
        const uint8_t* a = align16_down(src);
        const uint32_t bytes = round16((uint32_t)(src - a) + (uint32_t)n * (uint32_t)p.rb);
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        tma_load_1d(ring + (size_t)s * p.stage_bytes, a, bytes, &full_bar[s], pol);
      }
      if (!ok) {
        if (p.err) atomicOr(p.err, kErrTimeout);
        // the copies already issued land before the CTA may exit (bounded)
        for (int j = (i > p.nstage ? i - p.nstage : 0); j < i; ++j)
          mbar_wait_spin(&full_bar[j % p.nstage], (uint32_t)(j / p.nstage) & 1u, kLinWaitNs);
      }
    }
    return;
  }

  // ---------------- consumers: q8_1 of x, once, into shared memory
  const int T = p.T, K = p.K, nbk = K / 32;
  int8_t* aq = reinterpret_cast<int8_t*>(lin_smem);
  float* ad = reinterpret_cast<float*>(lin_smem + (size_t)T * K);
  int* as = reinterpret_cast<int*>(ad + (size_t)T * nbk);
  for (int b = tid; b < T * nbk; b += kLinConsumers) {
    const int t = b / nbk, kb = b - t * nbk;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * K + 32 * kb);
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[8];
      bf16x8_to_f32(__ldg(src + i), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * i + j] = f[j];
    }
    uint32_t qw[8];
    float d;
    int sum;
    q8_1_quantize_block(v, qw, d, sum);
    uint4* dq = reinterpret_cast<uint4*>(aq + (size_t)t * K + 32 * kb);
    dq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    dq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    ad[b] = f16_bits_to_f32(f32_to_f16_bits_rn(d));   // the dot uses the stored fp16 scale
    as[b] = sum;
  }
  consumer_sync<kLinConsumers>();

  ActSrc act;
  act.q = aq; act.d = ad; act.s = as; act.xb = nullptr; act.xf = nullptr; act.n = K;
  bool ok = true;
  for (int i = 0; i < nst; ++i) {
    const int s = i % p.nstage;
    if (!lin_wait(&full_bar[s], (uint32_t)(i / p.nstage) & 1u, abort)) {
      ok = false;
      break;
    }
    const int r0 = r_begin + i * p.rps;
    const int n = min(p.rps, r_end - r0);
    const uint8_t* src = p.rows + (size_t)r0 * p.rb;
    const uint8_t* base = ring + (size_t)s * p.stage_bytes + (src - align16_down(src));
    for (int j = warp; j < n; j += kLinConsumerWarps) {
      const uint8_t* row = base + (size_t)j * p.rb;
      float acc[LT];
#pragma unroll
      for (int t = 0; t < LT; ++t) acc[t] = 0.f;
      for (int b = lane; b < nbk; b += 32) {
        ActQ8 a[LT];
#pragma unroll
        for (int t = 0; t < LT; ++t)
          if (LT == 1 || t < T) a[t] = act_block(act, t, b);
        accum_q_block<WT, LT>(row, K, b, a, T, acc);
      }
#pragma unroll
      for (int t = 0; t < LT; ++t)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
      float v = acc[0];
#pragma unroll
      for (int t = 1; t < LT; ++t)
        if (lane == t) v = acc[t];
      if (lane < T) {
        const int rn = r0 + j;
        const float rs = p.row_scale ? __ldg(p.row_scale + rn) : 1.0f;
        p.out[(size_t)lane * p.N + rn] = (uint16_t)f32_to_bf16_bits_rn(v * rs);
      }
    }
    mbar_arrive(&empty_bar[s]);
  }
  if (!ok && p.err) atomicOr(p.err, kErrTimeout);
}

template <int WT, int LT>
cudaError_t launch_lin_t(const LinParams& p, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(k_linear<WT, LT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_linear<WT, LT><<<grid, kLinThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int WT>
cudaError_t launch_lin_w(const LinParams& p, int grid, size_t smem, cudaStream_t stream) {
  return p.T == 1 ? launch_lin_t<WT, 1>(p, grid, smem, stream) : launch_lin_t<WT, 8>(p, grid, smem, stream);
}

}  // namespace

// Shared-memory plan: q8_1 activations, then as many row slots (2..6 of
// about 24 KB, whole rows) as fit in the 227 KB a CTA may use.
bool plan_linear(LinParams& p) {
  constexpr size_t kSmemMax = 227 * 1024 - 512;   // static shared memory of the kernel stays below 512 B
  if (p.T < 1 || p.T > kLinearMaxT || p.N < 1 || p.rb <= 0) return false;
  const size_t act = ((size_t)p.T * p.K + 8 * (size_t)p.T * (p.K / 32) + 127) & ~size_t(127);
  if (act >= kSmemMax) return false;
  const int G = sm_count();
  const int rows_cta = (p.N + G - 1) / G;
  int rps = (int)((24 * 1024) / (size_t)p.rb);
  if (rps < 1) rps = 1;
  if (rps > rows_cta) rps = rows_cta;
  const size_t sb = (((size_t)rps * p.rb + 32) + 127) & ~size_t(127);
  const size_t room = kSmemMax - act;
  int ns = (int)(room / sb);
  if (ns > 6) ns = 6;
  if (ns < 2) return false;
  p.act_bytes = (int)act;
  p.rps = rps;
  p.stage_bytes = (int)sb;
  p.nstage = ns;
  p.grid = G < p.N ? G : p.N;
  return true;
}

size_t linear_smem_bytes(const LinParams& p) { return (size_t)p.act_bytes + (size_t)p.nstage * p.stage_bytes; }

cudaError_t launch_linear(const LinParams& p, cudaStream_t stream) {
  const size_t smem = linear_smem_bytes(p);
  switch (p.type) {
    case W_NVFP4:
      if (p.rb % 16 != 0) return launch_lin_w<W_NVFP4_U>(p, p.grid, smem, stream);
      return launch_lin_w<W_NVFP4>(p, p.grid, smem, stream);
    case W_Q4_K: return launch_lin_w<W_Q4_K>(p, p.grid, smem, stream);
    case W_Q8_0: return launch_lin_w<W_Q8_0>(p, p.grid, smem, stream);
    case W_Q6_K: return launch_lin_w<W_Q6_K>(p, p.grid, smem, stream);
    case W_Q4_0: return launch_lin_w<W_Q4_0>(p, p.grid, smem, stream);
    case W_Q4_1: return launch_lin_w<W_Q4_1>(p, p.grid, smem, stream);
    case W_Q5_0: return launch_lin_w<W_Q5_0>(p, p.grid, smem, stream);
    case W_Q5_1: return launch_lin_w<W_Q5_1>(p, p.grid, smem, stream);
    case W_Q5_K: return launch_lin_w<W_Q5_K>(p, p.grid, smem, stream);
    case W_MXFP4: return launch_lin_w<W_MXFP4>(p, p.grid, smem, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qre
