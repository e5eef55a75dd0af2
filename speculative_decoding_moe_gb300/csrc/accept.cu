// accept.cu -- vocab-parallel argmax and greedy prefix acceptance.
//
// "Speculating on a Strix Halo", section "Speculative decoding": under greedy
// decoding the target accepts only tokens it would have produced itself, and a
// cycle commits the accepted draft prefix plus one token of the target's own.
// Part 2, section "Why drafter performance doesn't really matter": the n-th
// draft is accepted only if the n-1 before it were.
//
// Grid = (k+1) rows x `chunks` vocabulary slices.  Each CTA reduces its slice
// to one 64-bit key (monotone float key << 32 | ~column), so the maximum key is
// the largest logit with the lowest column among equals.  The last CTA to
// finish (atomic ticket, no waiting) reduces the slices of every row, matches
// the draft prefix and writes tau and the committed tokens.
#include <map>
#include <mutex>

#include "dfv_internal.cuh"

namespace dfv {

constexpr int kAcceptThreads = 256;

__device__ __forceinline__ unsigned long long pack_key(float v, int col) {
  return ((unsigned long long)float_key(v) << 32) | (unsigned long long)(0xffffffffu - (unsigned)col);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(AcceptParams p) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x / p.chunks, ch = blockIdx.x % p.chunks;
  const long long V = p.V;
  const long long span = (((V + p.chunks - 1) / p.chunks) + 7) & ~7ll;  // multiple of 8 keeps 16-byte loads aligned
  const long long v0 = min(V, ch * span), v1 = min(V, v0 + span);
  unsigned long long best = 0ull;

  if (p.dtype == DFV_BF16) {
    const uint16_t *lg = reinterpret_cast<const uint16_t *>(p.logits) + (size_t)row * V;
    if ((V % 8) == 0 && (v0 % 8) == 0) {
      for (long long v = v0 + 8 * threadIdx.x; v < v1; v += 8 * kAcceptThreads) {
        if (v + 8 <= v1) {
          const uint4 u = ldg_stream(lg + v);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            best = umax64(best, pack_key(bf16_lo(w[q]), (int)(v + 2 * q)));
            best = umax64(best, pack_key(bf16_hi(w[q]), (int)(v + 2 * q + 1)));
          }
        } else {
          for (long long j = v; j < v1; ++j) best = umax64(best, pack_key(__uint_as_float((uint32_t)lg[j] << 16), (int)j));
        }
      }
    } else {
      for (long long v = v0 + threadIdx.x; v < v1; v += kAcceptThreads)
        best = umax64(best, pack_key(__uint_as_float((uint32_t)lg[v] << 16), (int)v));
    }
  } else {
    const float *lg = reinterpret_cast<const float *>(p.logits) + (size_t)row * V;
    if ((V % 4) == 0 && (v0 % 4) == 0) {
      for (long long v = v0 + 4 * threadIdx.x; v < v1; v += 4 * kAcceptThreads) {
        if (v + 4 <= v1) {
          const uint4 u = ldg_stream(lg + v);
          best = umax64(best, pack_key(__uint_as_float(u.x), (int)v));
          best = umax64(best, pack_key(__uint_as_float(u.y), (int)v + 1));
          best = umax64(best, pack_key(__uint_as_float(u.z), (int)v + 2));
          best = umax64(best, pack_key(__uint_as_float(u.w), (int)v + 3));
        } else {
          for (long long j = v; j < v1; ++j) best = umax64(best, pack_key(lg[j], (int)j));
        }
      }
    } else {
      for (long long v = v0 + threadIdx.x; v < v1; v += kAcceptThreads) best = umax64(best, pack_key(lg[v], (int)v));
    }
  }

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
  __shared__ unsigned long long s_w[kAcceptThreads / 32];
  __shared__ unsigned s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s_w[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int w = 0; w < kAcceptThreads / 32; ++w) b = umax64(b, s_w[w]);
    p.partial[blockIdx.x] = b;
    __threadfence();
    s_last = (atomicAdd(p.cnt, 1u) == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int s_a[kMaxBlock + 1];
  const int rows = p.k + 1;
  for (int r = warp; r < rows; r += kAcceptThreads / 32) {
    unsigned long long b = 0ull;
    for (int c = lane; c < p.chunks; c += 32) b = umax64(b, __ldcg(p.partial + r * p.chunks + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b = umax64(b, __shfl_xor_sync(0xffffffffu, b, o));
    if (lane == 0) s_a[r] = (int)(0xffffffffu - (unsigned)(b & 0xffffffffull));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < p.k && p.draft[n] == s_a[n]) ++n;
    *p.tau = n + 1;
    if (p.committed)
      for (int i = 0; i <= p.k; ++i) p.committed[i] = (i <= n) ? s_a[i] : -1;
    *p.cnt = 0u;
  }
}

cudaError_t launch_accept(const AcceptParams &p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.k + 1) * p.chunks);
  cfg.blockDim = dim3(kAcceptThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_kernel, p);
}

}  // namespace dfv

// ----------------------------------------------------------------------------
// Allocation-free variant of the acceptance launch.
//
// Some callers cannot allocate device memory: a runtime that hands the
// library a fixed memory budget, a caller that owns no allocator (plain C host
// code without access to the framework's caching allocator), or code that must
// not call cudaMalloc on its path.  For them the acceptance kernel's scratch
// (one 64-bit partial per CTA plus the last-CTA ticket) lives in this
// file-scope device array instead of a caller-provided workspace.  Every GPU
// that loads the library keeps the array (about 41 KB) until the process
// exits.  All calls share it: calls whose kernels overlap on the GPU race, so
// such calls must be ordered (one stream, or synchronised).
namespace dfv {
namespace {
constexpr int kNoAllocMaxChunks = 304;
constexpr size_t kNoAllocPartials = (size_t)(kMaxBlock + 1) * kNoAllocMaxChunks;
// [0, 32): ticket counter (first 4 bytes); [32, 32 + kNoAllocPartials): partials
static __device__ __align__(256) unsigned long long g_accept_scratch[32 + kNoAllocPartials];

std::mutex g_scratch_mu;
// device address of the array, per CUDA context: the address belongs to the
// context that loaded the module, so a new context (another device, or the
// primary context again after cudaDeviceReset) gets its own lookup
std::map<CUcontext, void *> g_scratch_ptr;

CUresult current_context(CUcontext *ctx) {
  using Fn = CUresult (*)(CUcontext *);
  static Fn fn = nullptr;
  static bool tried = false;
  if (!tried) {  // called with g_scratch_mu held
    tried = true;
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
    else
      cudaGetLastError();
  }
  return fn ? fn(ctx) : CUDA_ERROR_NOT_FOUND;
}
}  // namespace

cudaError_t accept_noalloc_scratch(void **out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CUcontext ctx = nullptr;
  if (current_context(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx) {
    auto it = g_scratch_ptr.find(ctx);
    if (it != g_scratch_ptr.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  // The array's name is only a host-side stand-in: the device address of the
  // current context's copy has to be looked up with that context current.  The
  // lookup also creates the device's primary context when none is current yet.
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_accept_scratch);
  if (e != cudaSuccess) return e;
  if (!ctx && (current_context(&ctx) != CUDA_SUCCESS || !ctx)) return cudaErrorDeviceUninitialized;
  g_scratch_ptr[ctx] = ptr;
  *out = ptr;
  return cudaSuccess;
}

int accept_noalloc_max_chunks() { return kNoAllocMaxChunks; }
}  // namespace dfv
