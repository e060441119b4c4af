// Prompt-path (prefill) kernels on the sm_103a tensor cores.
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "tc.cuh"

namespace qre {

// ------------------------------------------------------------------ tensor-core check

// D[128][N] = A[128][K] * B[N][K]^T, fp16 inputs (row-major), fp32 out, on
// the tensor cores: one CTA of 4 warps stages 64-wide K slices of A and B
// into swizzled shared-memory tiles, one thread issues four kind::f16 MMAs
// per slice into tensor memory, the warps read their 32 lanes back.
__global__ void __launch_bounds__(128, 1) k_tc_gemm_check(const uint16_t* A, const uint16_t* B, int K, int N,
                                                           float* D, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sa = base;
  uint8_t* sb = base + 16384;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = tc::idesc_f16(128, (uint32_t)N, false);
  uint32_t phase = 0;
  bool ok = true;
  for (int k0 = 0; k0 < K; k0 += 64) {
    for (int i = tid; i < 128 * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(sa + tc::sw128_chunk(r, c)) =
          *reinterpret_cast<const uint4*>(A + (size_t)r * K + k0 + 8 * c);
    }
    for (int i = tid; i < N * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(sb + tc::sw128_chunk(r, c)) =
          *reinterpret_cast<const uint4*>(B + (size_t)r * K + k0 + 8 * c);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_f16(tmem, tc::desc_sw128(smem_addr(sa) + 32 * kk), tc::desc_sw128(smem_addr(sb) + 32 * kk), idesc,
                    (k0 > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&bar);
    }
    if (!mbar_wait_bounded(&bar, phase, kWaitLimit)) ok = false;
    phase ^= 1u;
    tc::fence_after_sync();
  }
  for (int j0 = 0; j0 < N; j0 += 32) {
    uint32_t r[32];
    tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)j0, r);
    tc::tmem_ld_wait();
    const int m = 32 * warp + (tid & 31);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j0 + j < N) D[(size_t)m * N + j0 + j] = __uint_as_float(r[j]);
  }
  if (!ok) atomicOr(err, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_tc_gemm_check(const uint16_t* A, const uint16_t* B, int K, int N, float* D, int* err,
                                 cudaStream_t stream) {
  const size_t smem = 1024 + 16384 + (size_t)N * 128;
  cudaError_t e = cudaFuncSetAttribute(k_tc_gemm_check, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_tc_gemm_check<<<1, 128, smem, stream>>>(A, B, K, N, D, err);
  return cudaGetLastError();
}

}  // namespace qre
