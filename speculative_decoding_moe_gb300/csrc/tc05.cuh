// tc05.cuh -- fifth-generation tensor-core (tcgen05) building blocks for
// sm_100-family GPUs, written as inline PTX: tensor-memory (TMEM)
// allocation, the shared-memory matrix descriptor of a K-major operand tile
// stored with the 128-byte swizzle (the layout a TMA copy with
// CU_TENSOR_MAP_SWIZZLE_128B writes), the instruction descriptor of a dense
// bf16 x bf16 -> fp32 MMA, the MMA itself, its commit to an mbarrier, and the
// TMEM -> register loads of the epilogue.
//
// Operand layout (K-major, bf16): row r of a tile holds 64 consecutive K
// elements (128 bytes); the 16-byte chunk j of row r sits at chunk j ^ (r & 7)
// (the 128-byte swizzle), rows at a 128-byte pitch, so eight rows form one
// 1024-byte swizzle atom.  A tile's base must be 1024-byte aligned.
#pragma once

#include "dfv_internal.cuh"

namespace dfv {
namespace {

// ---------------------------------------------------------------- TMEM
// One warp allocates `ncols` (a power of two, 32..512) TMEM columns of all 128
// lanes and writes their base address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle:
// start address (bits 0-13, in 16-byte units), leading-dimension byte offset
// (bits 16-29; unused by this layout, set to 1), stride byte offset between
// 8-row groups (bits 32-45: 1024 bytes), descriptor version 1 (bits 46-47),
// layout type 2 = 128-byte swizzle (bits 61-63).  Advancing K by 16 elements
// (32 bytes) inside the 128-byte atom adds 2 to the start address field.
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3fffu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both
// operands K-major, no negation or sparsity: D format (bits 4-5) = 1 (f32),
// A format (bits 7-9) = 1 (bf16), B format (bits 10-12) = 1 (bf16),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).  M = 128 takes N in 16..256,
// multiples of 16.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one thread issues.  accumulate = 0 writes D.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier at `bar` receives one arrival once every MMA this thread issued
// before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Lane l of warp w reads TMEM lane 32 (w % 4) + l, 16 consecutive fp32
// columns from `taddr` (the column in bits 0-15, the lane in bits 16-31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (r, k) (k < 64) of a K-major 128-byte-swizzled bf16
// tile: row pitch 128 bytes, 16-byte chunk k / 8 XOR r % 8.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
  return (uint32_t)r * 128u + ((((uint32_t)k >> 3) ^ ((uint32_t)r & 7u)) << 4) + (((uint32_t)k & 7u) << 1);
}

}  // namespace
}  // namespace dfv
