// ffn_common.cuh -- pieces shared by the multi-launch expert FFN kernels
// (bf16/fp32 weights in ffn.cu, mxfp4 weights in ffn_mxfp4.cu): the unit
// partition, the down-tile ticket with the slot-ordered combine, and the host
// launch / occupancy helpers.
#pragma once

#include <map>
#include <mutex>
#include <utility>

#include "dfv_internal.cuh"

namespace dfv {
namespace {

// Contiguous share [lo, hi) of U units for this CTA.
__device__ __forceinline__ void unit_range(int U, int &lo, int &hi) {
  lo = (int)(((long long)blockIdx.x * U) / gridDim.x);
  hi = (int)(((long long)(blockIdx.x + 1) * U) / gridDim.x);
}

// out[t][r] = residual[t][r] + sum_s ys[t*K+s][r], slot order, + ys[k*K+t][r]
// (shared expert, when ns) for the rows of down tile dt (kDownTile rows).
// Called by the last unit to finish that tile.
__device__ __forceinline__ void combine_tile(const FfnParams &p, int dt) {
  const int r0 = dt * kDownTile;
  const int rows = min(kDownTile, p.d - r0);
  for (int idx = threadIdx.x; idx < p.k * kDownTile; idx += blockDim.x) {
    const int t = idx / kDownTile, rr = idx % kDownTile;
    if (rr >= rows) continue;
    const int r = r0 + rr;
    float s = 0.f;
    for (int sl = 0; sl < p.K; ++sl) s += __ldcg(p.ws.ys + (size_t)(t * p.K + sl) * p.d + r);
    if (p.ns) s += __ldcg(p.ws.ys + (size_t)(p.k * p.K + t) * p.d + r);
    if (p.residual) s = load_act(p.residual, (size_t)t * p.d + r, p.act) + s;
    store_act(p.out, (size_t)t * p.d + r, p.act, s);
  }
}

// Ticket for tile dt after this CTA wrote its ys rows of that tile; the unit
// that arrives last (of nW, one per woken expert, the shared one included)
// runs the combine and returns
// the ticket to zero.  Nothing waits.
__device__ __forceinline__ void finish_down_unit(const FfnParams &p, int dt, int nW) {
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(p.ws.down_cnt + dt, 1u) == (unsigned)(nW - 1)) ? 1u : 0u;
  __syncthreads();
  if (s_last) {
    __threadfence();
    combine_tile(p, dt);
    __syncthreads();
    if (threadIdx.x == 0) p.ws.down_cnt[dt] = 0u;
  }
}

// ---------------------------------------------------------------- host side
template <typename F>
cudaError_t launch_ffn_kernel(F kern, int grid, int threads, size_t smem, const FfnParams &p, cudaStream_t s,
                              bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Raise a kernel's dynamic shared-memory limit once per (device, kernel); later
// calls (including ones made while a stream is being captured) only look up.
// Any request above 32 KB sets it: the 48 KB that needs no opt-in counts the
// kernel's static shared memory too, so a request just under 48 KB can still
// need it (the mxfp4 down kernel at d_ff = 1536 asks for exactly 48 KB).
template <typename F>
cudaError_t ensure_smem(F kern, size_t bytes) {
  if (bytes <= 32 * 1024) return cudaSuccess;
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(dev, (const void *)kern);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

// CTAs of `kern` that fit on the whole GPU at once (0 when none fits).
template <typename F>
int occupancy_grid(F kern, int threads, size_t smem) {
  int dev = 0, sms = 0, per = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ensure_smem(kern, smem) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, threads, smem) != cudaSuccess) return 0;
  return sms * per;
}

}  // namespace
}  // namespace dfv
