// mxfp4_common.cuh -- widening of mxfp4 codes (E2M1) to fp16 MMA operands,
// and the fp16 staging of activation rows with a per-row power-of-two scale.
// Shared by the multi-launch (ffn_mxfp4.cu) and the single-launch block-scaled
// (layer_fused_bs.cu) kernels; both apply each block's E8M0 scale to the fp32
// partial sum of that block's MMAs.
//
// OCP Microscaling Formats (MX) v1.0, as used by the MI355X / vLLM write-up
// (allbreaknews.com/?p=4397), section "Why Quantize the Target Model on Top?":
// an element is a 4-bit E2M1 code (sign, 2 exponent bits with bias 1, 1
// mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) and every 32
// consecutive elements of a row share one E8M0 scale 2^(s - 127).
#pragma once

#include "dfv_internal.cuh"

namespace dfv {
namespace {

// One scale byte (kept in L1: the four chunks of a sector share it).
__device__ __forceinline__ uint32_t ldg_scale(const uint8_t *p) {
  uint32_t v;
  asm("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Four bytes of codes -> four fp16x2, byte b -> r[b], low nibble in the low half.
__device__ __forceinline__ void e2m1_word(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 q0, q1, q2, q3;\n mov.b32 {q0, q1, q2, q3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, q0;\n cvt.rn.f16x2.e2m1x2 %1, q1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, q2;\n cvt.rn.f16x2.e2m1x2 %3, q3;\n}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_f16x(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Power-of-two exponent that brings a row's largest magnitude amax into
// [1, 2): a block's fp32 partial sum then stays near the true sum, so its
// scale 2^(s-127) cannot push it past the fp32 range short of the true
// result itself.
__device__ __forceinline__ int row_shift(float amax) {
  if (!(amax > 0.f) || !(amax < INFINITY)) return 0;
  int ex;
  frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
  return min(max(1 - ex, -126), 126);
}

__device__ __forceinline__ float exp2i(int s) { return __int_as_float((127 + s) << 23); }

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace
}  // namespace dfv
