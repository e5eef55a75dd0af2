// router.cu -- fused MoE router for a block of k positions.
//
// "Speculating on a Strix Halo", section "What the pieces cost": every token of
// the verify block routes to its own experts, so the block wakes the union of
// its rows' top-K sets; section "The verify's own cost": tokens are sorted by
// expert before the grouped expert launch.
//
// One launch does all of it:
//   1. (optional) RMSNorm of each row, rounded to the activation dtype;
//   2. router GEMV, one CTA per expert: logits[t][e] = x[t] . Wr[e] in fp32,
//      in a fixed summation order;
//   3. the last CTA to finish (atomic ticket, no waiting) takes the top-K of
//      every row with a warp per row (redux.sync max on monotone float keys,
//      ties to the lowest expert id), the routing weights, the woken-expert
//      union (ascending), per-expert pair offsets (block-wide exclusive scan)
//      and the pair gather list sorted by (expert, token).  With an always-on
//      shared expert (same section) it closes the workspace tables with that
//      expert: id E, one pair k*K + t per row, weight 1.
#include "dfv_internal.cuh"

namespace dfv {

// The GEMV and the row norms run on the first kGemvThreads threads, in a
// fixed summation order.  A launch has 256 threads for k <= 8 and 512 above,
// so the top-K tail gives every row of a block its own warp; the arithmetic
// of a row is the same in both.
constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// Fixed-order block sum of v[0..n) over the GEMV warps: warp butterfly, then
// warps in index order.  Result in out[0..n) (shared), visible after the
// trailing __syncthreads.
template <int N>
__device__ __forceinline__ void block_sum_rows(float (&v)[N], int n, float (*red)[N], float *out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < N; ++t) {
    if (t < n) {
      float a = v[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(kFull, a, o);
      v[t] = a;
    }
  }
  if (lane == 0 && warp < kGemvWarps) {
#pragma unroll
    for (int t = 0; t < N; ++t)
      if (t < n) red[warp][t] = v[t];
  }
  __syncthreads();
  if (threadIdx.x < n) {
    float a = 0.f;
    for (int w = 0; w < kGemvWarps; ++w) a += red[w][threadIdx.x];
    out[threadIdx.x] = a;
  }
  __syncthreads();
}

// Eight consecutive activation / router-weight elements as floats.
__device__ __forceinline__ void load8(const void *base, size_t elem, int dt, float (&f)[8]) {
  if (dt == DFV_BF16) {
    uint4 u = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(base) + elem);
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  } else {
    const float4 *q = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + elem);
    float4 a = q[0], b = q[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

__device__ __forceinline__ float round_act(float v, int act) {
  return act == DFV_BF16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// Top-K of one row of E logits by one warp.  Lane l owns experts
// [l*epl, (l+1)*epl) (blocked), sorted locally by (key desc, id asc); each of
// the K rounds takes the warp maximum of the lane heads and the lowest lane
// holding it, which is the lowest expert id among equal logits.
__device__ void topk_row(const float *lg, int E, int K, int32_t *idx_out, float *sel_out) {
  const int lane = threadIdx.x & 31;
  const int epl = (E + 31) >> 5;  // <= 8
  uint32_t key[8];
  int id[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    int e = lane * epl + q;
    bool ok = (q < epl) && (e < E);
    key[q] = ok ? max(float_key(lg[e]), 1u) : 0u;  // 0 only for empty slots
    id[q] = ok ? e : 0x7fffffff;
  }
  // stable descending bubble sort of 8 (strict compare keeps lower ids first)
#pragma unroll
  for (int i = 0; i < 7; ++i) {
#pragma unroll
    for (int j = 0; j < 7 - i; ++j) {
      if (key[j + 1] > key[j]) {
        uint32_t tk = key[j]; key[j] = key[j + 1]; key[j + 1] = tk;
        int ti = id[j]; id[j] = id[j + 1]; id[j + 1] = ti;
      }
    }
  }
  for (int s = 0; s < K; ++s) {
    uint32_t m = __reduce_max_sync(kFull, key[0]);
    unsigned b = __ballot_sync(kFull, key[0] == m);
    int src = __ffs(b) - 1;
    int win = __shfl_sync(kFull, id[0], src);
    if (lane == 0) {
      idx_out[s] = win;
      sel_out[s] = lg[win];
    }
    if (lane == src) {
#pragma unroll
      for (int q = 0; q < 7; ++q) { key[q] = key[q + 1]; id[q] = id[q + 1]; }
      key[7] = 0u;
      id[7] = 0x7fffffff;
    }
  }
}

template <int kRouterThreads>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(RouterParams p) {
  constexpr int kRouterWarps = kRouterThreads / 32;
  pdl_trigger();
  // this CTA's router row does not depend on the previous launch: start its
  // fetch into L2 before waiting for that launch to finish
  if (threadIdx.x == 0) {
    const size_t rb = (size_t)p.d * (p.rdt == DFV_BF16 ? 2 : 4);
    prefetch_l2(reinterpret_cast<const char *>(p.wr) + (size_t)blockIdx.x * rb, (uint32_t)rb);
  }
  pdl_wait();  // x may be the previous layer's output

  __shared__ float s_red[kGemvWarps][kMaxBlock];
  __shared__ float s_inv[kMaxBlock];
  __shared__ float s_dot[kMaxBlock];
  __shared__ unsigned s_last;

  const int tid = threadIdx.x;
  const int k = p.k, d = p.d, E = p.E, K = p.K;
  const int e = blockIdx.x;

  // bf16 activations: the k rows' pieces of one column chunk are all loaded
  // before any arithmetic, so their latencies overlap (the sums below keep
  // the generic path's order exactly)
  const bool xbf = p.act == DFV_BF16;
  auto load_rows = [&](int c, uint4 (&xv)[kMaxBlock]) {
#pragma unroll
    for (int t = 0; t < kMaxBlock; ++t)
      xv[t] = t < k ? __ldcg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.x) +
                                                             (size_t)t * d + (size_t)c * 8))
                    : make_uint4(0u, 0u, 0u, 0u);
  };
  auto unpack = [](const uint4 &v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  };

  // ---- 1. RMSNorm scale per row (fixed-order sums)
  if (p.fuse_norm) {
    float ss[kMaxBlock];
#pragma unroll
    for (int t = 0; t < kMaxBlock; ++t) ss[t] = 0.f;
    for (int c = tid < kGemvThreads ? tid : d; c < d / 8; c += kGemvThreads) {
      if (xbf) {
        uint4 xv[kMaxBlock];
        load_rows(c, xv);
#pragma unroll
        for (int t = 0; t < kMaxBlock; ++t) {
          if (t < k) {
            float f[8];
            unpack(xv[t], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) ss[t] = fmaf(f[q], f[q], ss[t]);
          }
        }
        continue;
      }
#pragma unroll
      for (int t = 0; t < kMaxBlock; ++t) {
        if (t < k) {
          float f[8];
          load8(p.x, (size_t)t * d + c * 8, p.act, f);
#pragma unroll
          for (int q = 0; q < 8; ++q) ss[t] = fmaf(f[q], f[q], ss[t]);
        }
      }
    }
    block_sum_rows<kMaxBlock>(ss, k, s_red, s_inv);
    if (tid < k) s_inv[tid] = 1.0f / sqrtf(s_inv[tid] / (float)d + p.eps);
    __syncthreads();
  }

  // ---- 2. GEMV for expert e
  float acc[kMaxBlock];
#pragma unroll
  for (int t = 0; t < kMaxBlock; ++t) acc[t] = 0.f;
  for (int c = tid < kGemvThreads ? tid : d; c < d / 8; c += kGemvThreads) {
    float w[8];
    load8(p.wr, (size_t)e * d + c * 8, p.rdt, w);
    if (xbf) {
      uint4 xv[kMaxBlock];
      load_rows(c, xv);
#pragma unroll
      for (int t = 0; t < kMaxBlock; ++t) {
        if (t < k) {
          float f[8];
          unpack(xv[t], f);
          if (p.fuse_norm) {
            const float inv = s_inv[t];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = round_act(f[q] * inv, DFV_BF16);
            if (e == 0) {
#pragma unroll
              for (int q = 0; q < 8; ++q) store_act(p.ws.xn, (size_t)t * d + c * 8 + q, DFV_BF16, f[q]);
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[t] = fmaf(f[q], w[q], acc[t]);
        }
      }
      continue;
    }
#pragma unroll
    for (int t = 0; t < kMaxBlock; ++t) {
      if (t < k) {
        float f[8];
        load8(p.x, (size_t)t * d + c * 8, p.act, f);
        if (p.fuse_norm) {
          const float inv = s_inv[t];
#pragma unroll
          for (int q = 0; q < 8; ++q) f[q] = round_act(f[q] * inv, p.act);
          if (e == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) store_act(p.ws.xn, (size_t)t * d + c * 8 + q, p.act, f[q]);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t] = fmaf(f[q], w[q], acc[t]);
      }
    }
  }
  block_sum_rows<kMaxBlock>(acc, k, s_red, s_dot);
  if (tid < k) p.ws.logits[(size_t)tid * E + e] = s_dot[tid];

  // ---- ticket: the last CTA finalises the routing
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(p.ws.router_cnt, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ float s_lg[kMaxBlock * kMaxExperts];
  __shared__ int32_t s_idx[kMaxBlock * kMaxTopK];
  __shared__ float s_sel[kMaxBlock * kMaxTopK];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ unsigned s_mask[kMaxBlock][kMaxExperts / 32];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_wsum[kRouterWarps], s_csum[kRouterWarps];

  for (int i = tid; i < k * E; i += kRouterThreads) s_lg[i] = __ldcg(p.ws.logits + i);
  for (int i = tid; i < kMaxExperts; i += kRouterThreads) s_cnt[i] = 0;
  for (int i = tid; i < kMaxBlock * (kMaxExperts / 32); i += kRouterThreads) (&s_mask[0][0])[i] = 0u;
  __syncthreads();

  const int lane = tid & 31, warp = tid >> 5;
  for (int t = warp; t < k; t += kRouterWarps) {
    topk_row(s_lg + t * E, E, K, s_idx + t * K, s_sel + t * K);
    __syncwarp();
    // routing weights: softmax restricted to the K selected (renormalised),
    // or the full softmax probability of each selected expert.  Lane s takes
    // selection s; the denominator is the warp's butterfly sum of the lanes'
    // terms (lane l's term sums experts l, l + 32, ... in that order)
    const float m0 = s_sel[t * K];
    const float z = lane < K ? expf(s_sel[t * K + lane] - m0) : 0.f;
    float den = 0.f;
    if (p.norm_topk) {
      den = z;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (lane + 32 * q < E) den += expf(s_lg[t * E + lane + 32 * q] - m0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    __syncwarp();
    if (lane < K) s_sel[t * K + lane] = z / den;
  }
  __syncthreads();

  for (int q = tid; q < k * K; q += kRouterThreads) {
    const int t = q / K, ex = s_idx[q];
    atomicAdd(&s_cnt[ex], 1);
    atomicOr(&s_mask[t][ex >> 5], 1u << (ex & 31));
  }
  __syncthreads();

  // block-wide exclusive scans over experts: woken position and pair offset
  int flag = 0, cnt = 0;
  if (tid < E) { cnt = s_cnt[tid]; flag = cnt > 0; }
  int fi = flag, ci = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int a = __shfl_up_sync(kFull, fi, o), b = __shfl_up_sync(kFull, ci, o);
    if (lane >= o) { fi += a; ci += b; }
  }
  if (lane == 31) { s_wsum[warp] = fi; s_csum[warp] = ci; }
  __syncthreads();
  int wbase = 0, cbase = 0, nW = 0;
  for (int w = 0; w < kRouterWarps; ++w) {
    if (w < warp) { wbase += s_wsum[w]; cbase += s_csum[w]; }
    nW += s_wsum[w];
  }
  const int wpos = wbase + fi - flag, off = cbase + ci - cnt;
  if (tid < E) s_off[tid] = off;
  if (flag) {
    p.ws.woken[wpos] = tid;
    p.ws.offsets[wpos] = off;
    if (p.u_woken) p.u_woken[wpos] = tid;
    if (p.u_offs) p.u_offs[wpos] = off;
  }
  if (tid == 0) {
    p.ws.offsets[nW] = k * K;
    *p.ws.n_woken = nW;
    if (p.u_offs) p.u_offs[nW] = k * K;
    if (p.u_nw) *p.u_nw = nW;
  }
  __syncthreads();

  for (int q = tid; q < k * K; q += kRouterThreads) {
    const int t = q / K, ex = s_idx[q];
    int rank = 0;
    for (int t2 = 0; t2 < t; ++t2) rank += (s_mask[t2][ex >> 5] >> (ex & 31)) & 1u;
    p.ws.gather[s_off[ex] + rank] = q;
    if (p.u_gather) p.u_gather[s_off[ex] + rank] = q;
    p.ws.topk_idx[q] = ex;
    p.ws.topk_w[q] = s_sel[q];
    if (p.u_idx) p.u_idx[q] = ex;
    if (p.u_w) p.u_w[q] = s_sel[q];
  }
  if (p.ns) {
    // the shared expert joins the workspace tables (not the caller's copies)
    // as the last woken expert, id E: every row selects it, pair k*K + t,
    // weight 1
    if (tid == 0) {
      p.ws.woken[nW] = E;
      p.ws.offsets[nW + 1] = k * K + k;
      *p.ws.n_woken = nW + 1;
    }
    for (int t = tid; t < k; t += kRouterThreads) {
      p.ws.gather[k * K + t] = k * K + t;
      p.ws.topk_w[k * K + t] = 1.f;
    }
  }
  if (tid == 0) *p.ws.router_cnt = 0u;
}

cudaError_t launch_router(const RouterParams &p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.E);
  const bool wide = p.k > 8;
  cfg.blockDim = dim3(wide ? 512 : 256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return wide ? cudaLaunchKernelEx(&cfg, router_kernel<512>, p) : cudaLaunchKernelEx(&cfg, router_kernel<256>, p);
}

}  // namespace dfv
