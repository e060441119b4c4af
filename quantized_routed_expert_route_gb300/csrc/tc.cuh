// Inline-PTX wrappers for the sm_103a tensor cores (tcgen05): tensor-memory
// allocation, shared-memory matrix descriptors, the kind::f16 MMA with fp32
// accumulation in tensor memory, its commit to an mbarrier, and tensor-memory
// loads for the epilogue.
//
// Operand layout used throughout: K-major tiles with the 128-byte swizzle.  A
// tile of R rows x 64 fp16 values occupies R * 128 bytes, rows 128 bytes apart,
// 8-row groups 1024 bytes apart, and inside each 1024-byte group the 16-byte
// chunk c of row r is stored at chunk position c ^ (r % 8).  Tile bases are
// 1024-byte aligned.  One MMA consumes K = 16 (32 bytes of each row); the k-th
// 16-wide step inside a 64-wide tile starts 32*k bytes into the tile.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace qre {
namespace tc {

// Byte offset of fp16 element (r, k) (k < 64) inside a swizzled tile.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t k) {
  const uint32_t lin = r * 128u + k * 2u;
  return lin ^ (((lin >> 7) & 7u) << 4);
}

// Byte offset of the 16-byte chunk c (elements 8c..8c+7) of row r.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                     // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;           // stride byte offset
  d |= (uint64_t)1u << 46;                     // version
  d |= (uint64_t)2u << 61;                     // SWIZZLE_128B
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, fp16 (or bf16) A
// and B, both K-major, M x N.
__host__ __device__ __forceinline__ uint32_t idesc_f16(uint32_t M, uint32_t N, bool bf16) {
  uint32_t d = 0;
  d |= 1u << 4;                       // D format: F32
  d |= (bf16 ? 1u : 0u) << 7;         // A format
  d |= (bf16 ? 1u : 0u) << 10;        // B format
  d |= (N >> 3) << 17;
  d |= (M >> 4) << 24;
  return d;
}

// Instruction descriptor of kind::mxf4nvf4 with block scaling (NVFP4: E2M1
// A and B, packed two values a byte, UE4M3 scales per 16 values along K),
// both K-major, fp32 accumulator, M x N.  Fields (the PTX ISA's descriptor
// for the block-scaled kinds): bits 4-5 the scale-B data id, 7-9 A format
// (E2M1 = 1 for the mxf4 kinds), 10-12 B format, 15/16 A/B major (0 =
// K-major), 17-22 N >> 3, 23 scale type (0 = UE4M3), 24-28 M >> 4, 29-30
// the scale-A data id.  With 16-value blocks an MMA (K = 64) uses four
// scales of a row, one 32-bit tensor-memory column: both data ids are 0.
__host__ __device__ __forceinline__ uint32_t idesc_mxf4nvf4(uint32_t M, uint32_t N) {
  uint32_t d = 0;
  d |= 1u << 7;                       // A: E2M1
  d |= 1u << 10;                      // B: E2M1
  d |= (N >> 3) << 17;
  d |= (M >> 4) << 24;                // scale type bit 23 = 0: UE4M3
  return d;
}

// Shared-memory descriptor of a plain (unswizzled) K-major tile whose 8-row
// groups of 16-byte rows are `sbo` bytes apart: the source of tcgen05.cp.
__device__ __forceinline__ uint64_t desc_plain(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                     // leading byte offset (one 16-byte column)
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32; // stride byte offset
  d |= (uint64_t)1u << 46;                     // version
  return d;                                    // swizzle 0: none
}

// 32 rows x 16 bytes of shared memory -> four consecutive 32-bit columns
// from `taddr` of tensor-memory lanes r, r+32, r+64, r+96 (row r to each of
// the four lane quarters).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= (A * scale_A) * (B * scale_B)^T with NVFP4 operands in shared
// memory and their per-16 UE4M3 scales in tensor memory (one column each for
// the 64 values of this MMA), issued by one thread.  Scale layout for M (or
// N) = 128 rows: four tensor-memory columns from sfa/sfb; column c of lane l
// holds the four scales (bytes, K order) of row (l % 32) + 32 c, the same in
// every lane quarter -- one 512-byte shared-memory atom (line r: rows r,
// r+32, r+64, r+96, four bytes each) copied by tmem_cp_32x128b_x4, or the
// same words stored by each lane quarter's warp with tmem_st16.
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Tensor memory: allocate `ncols` columns (a power of two >= 32) for the CTA;
// the whole warp executes it and the address lands in *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane (the warp
// reads lanes 32*(warp%4) .. +31; taddr carries the lane base in bits 16+).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Sixteen consecutive 32-bit columns of this thread's tensor-memory lane <- r
// (warp w writes lanes 32 * (w % 4) .. + 31; taddr carries that lane base).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// This thread's tensor-memory stores are complete.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Eight E2M1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// -> eight fp16 values as four f16x2 words (exact).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t codes, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
}

// Two UE4M3 bytes -> f16x2 (exact; bit 7 of each byte clear).
__device__ __forceinline__ uint32_t ue4m3x2_to_f16x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return h2;
}

// fp32 >= 0 -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_rne_sat(float v) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return (uint32_t)h & 0xFFu;
}

// Eight fp32 -> eight E2M1 codes (round to nearest even, saturating at 6,
// the sign kept), packed with element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8_rne_sat(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

}  // namespace tc
}  // namespace qre
