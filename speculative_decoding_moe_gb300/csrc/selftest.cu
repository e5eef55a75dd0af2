// selftest.cu -- runs the bounded waits of the single-launch kernels on
// conditions that never come true, so that a test can watch them give up,
// report and return (no counterpart on the method's pages).
//
// One CTA, one active thread: it waits on a shared-memory mbarrier phase that
// nobody completes, then on a grid barrier that a one-CTA launch can never
// fill.  Each wait is the production helper, with its production limit, so
// each gives up after about 2 s, sets its bit in the workspace error word and
// returns false.  No copy is issued, so nothing is in flight when a wait gives
// up, and the kernel exits normally.
#include "fused_common.cuh"
#include "mxfp4_common.cuh"

namespace dfv {

__global__ void __launch_bounds__(32) wait_selftest_kernel(const FusedParams p) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ volatile int s_abort;
  if (threadIdx.x != 0) return;
  s_abort = 0;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);  // one arrival completes phase 0; none is made
  mbar_init_fence();
  mbar_wait(b, 0u, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort);
  grid_sync(p, 2);  // needs 2 * gridDim.x = 2 arrivals; only this CTA arrives
  // the grid-barrier words back to zero, as a finished launch leaves them
  atomicExch(p.ws.sync, 0u);
  atomicExch(p.ws.sync + 1, 0u);
  atomicExch(p.ws.sync + 2, 0u);
}

cudaError_t launch_wait_selftest(const Workspace &w, cudaStream_t s) {
  FusedParams p = {};
  p.ws = w;
  wait_selftest_kernel<<<1, 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dfv

// ----------------------------------------------------------------------------
// The legacy-MMA fragment path of the expert kernels on one 16x16x16 product
// (no counterpart in the kernels' own work: it lets a test compare the tensor
// core's result with exact values).  "Speculating on a Strix Halo (part 2)",
// section "Two bugs upstream": a multiply-add whose only non-zero operands are
// one column of A and one row of B has an exact result, and a correct unit
// returns it whatever the sign of the zero operands.
//
// One warp computes D = A . B with the helpers and the operand mapping the
// expert kernels use: lane (g = lane / 4, c = lane % 4) holds rows g (M 0-7)
// and g + 8 (M 8-15) of A, and each 16-byte group of four consecutive columns
// 4c..4c+3 of a 16-column chunk feeds the MMA's k slots {2c, 2c+1} and
// {2c+8, 2c+9}; B's rows are read through the same permutation, so the sum
// over k is unchanged.  bf16 operands go through mma_bf16 (the bf16 kernels),
// fp16 operands through mma_f16x (the mxfp4 kernels).

namespace dfv {

__global__ void __launch_bounds__(32) mma_selftest_kernel(const uint16_t *A, const uint16_t *B, float *D, int bf16) {
  const int lane = threadIdx.x, g = lane >> 2, c = lane & 3;
  auto pair = [](uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); };
  // A rows g and g + 8, columns 4c..4c+3
  const uint32_t a0 = pair(A[g * 16 + 4 * c], A[g * 16 + 4 * c + 1]);
  const uint32_t a2 = pair(A[g * 16 + 4 * c + 2], A[g * 16 + 4 * c + 3]);
  const uint32_t a1 = pair(A[(g + 8) * 16 + 4 * c], A[(g + 8) * 16 + 4 * c + 1]);
  const uint32_t a3 = pair(A[(g + 8) * 16 + 4 * c + 2], A[(g + 8) * 16 + 4 * c + 3]);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int n = nt * 8 + g;  // output column this lane's B fragment feeds
    const uint32_t b0 = pair(B[(4 * c) * 16 + n], B[(4 * c + 1) * 16 + n]);
    const uint32_t b1 = pair(B[(4 * c + 2) * 16 + n], B[(4 * c + 3) * 16 + n]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (bf16)
      mma_bf16(acc, a0, a1, a2, a3, b0, b1);
    else
      mma_f16x(acc, a0, a1, a2, a3, b0, b1);
    const int j = nt * 8 + 2 * c;
    D[g * 16 + j] = acc[0];
    D[g * 16 + j + 1] = acc[1];
    D[(g + 8) * 16 + j] = acc[2];
    D[(g + 8) * 16 + j + 1] = acc[3];
  }
}

cudaError_t launch_mma_selftest(const void *A, const void *B, float *D, int bf16, cudaStream_t s) {
  mma_selftest_kernel<<<1, 32, 0, s>>>(static_cast<const uint16_t *>(A), static_cast<const uint16_t *>(B), D, bf16);
  return cudaGetLastError();
}

}  // namespace dfv
