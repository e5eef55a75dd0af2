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

// ----------------------------------------------------------------------------
// The tcgen05 path on one tile (no counterpart in the method: it lets a test
// check the shared-memory and instruction descriptors, the TMEM allocation and
// the epilogue loads against a plain matrix product before the batched expert
// kernels rely on them).  One CTA of four warps: the operands go to shared
// memory in the 128-byte-swizzled K-major layout, one thread issues K/16 MMAs
// into TMEM (M = 128 rows of A, N rows of B), commits them to an mbarrier, and
// each warp reads its 32 TMEM lanes back.  The wait is bounded (2 s); a
// timeout leaves status = 1.
#include "tc05.cuh"

namespace dfv {

__global__ void __launch_bounds__(128) tc05_selftest_kernel(const uint16_t *A, const uint16_t *B, int N, int K,
                                                            float *D, int *status) {
  extern __shared__ __align__(1024) unsigned char tsm_raw[];
  unsigned char *tsm = tsm_raw + ((1024u - (smem_u32(tsm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int natoms = K / 64;
  const uint32_t a_base = smem_u32(tsm), b_base = a_base + (uint32_t)natoms * 128u * 128u;
  // operands into the swizzled layout: atom a holds K columns [64a, 64a + 64)
  for (int i = tid; i < 128 * K; i += 128) {
    const int r = i / K, kk = i % K;
    *reinterpret_cast<uint16_t *>(tsm + (kk / 64) * 128 * 128 + sw128_off(r, kk % 64)) = A[i];
  }
  for (int i = tid; i < N * K; i += 128) {
    const int r = i / K, kk = i % K;
    *reinterpret_cast<uint16_t *>(tsm + natoms * 128 * 128 + (kk / 64) * N * 128 + sw128_off(r, kk % 64)) = B[i];
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> async-proxy reads
  const uint32_t bar = smem_u32(&s_bar);
  uint32_t ncols = 32;
  while ((int)ncols < N) ncols <<= 1;
  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar, 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(128, N);
    for (int ks = 0; ks < K / 16; ++ks) {
      const int at = ks / 4, kk = ks % 4;
      const uint64_t ad = sdesc_k128(a_base + (uint32_t)at * 128u * 128u) + (uint64_t)(2 * kk);
      const uint64_t bd = sdesc_k128(b_base + (uint32_t)at * (uint32_t)N * 128u) + (uint64_t)(2 * kk);
      tc_mma(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    tc_commit(bar);
  }
  __syncwarp();
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, 0u, (unsigned *)status, 1u, &s_abort);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) D[row * N + c0 + j] = v[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

cudaError_t launch_tc05_selftest(const void *A, const void *B, int N, int K, float *D, int *status, cudaStream_t s) {
  const size_t smem = 1024 + (size_t)(128 + N) * K * 2;
  cudaError_t e = cudaFuncSetAttribute(tc05_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc05_selftest_kernel<<<1, 128, smem, s>>>(static_cast<const uint16_t *>(A), static_cast<const uint16_t *>(B), N, K,
                                           D, status);
  return cudaGetLastError();
}

}  // namespace dfv
