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
