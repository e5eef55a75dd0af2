// fused_common.cuh -- pieces shared by the single-launch layer kernels
// (layer_fused.cu: bf16 experts; layer_fused_mxfp4.cu: mxfp4 experts): the
// thread layout, the bounded grid barrier and the routing prologue.
#pragma once

#include "dfv_internal.cuh"

namespace dfv {
namespace {

constexpr int kFW = 16;           // consumer warps
constexpr int kFC = kFW * 32;     // consumer threads
constexpr int kFT = kFC + 32;     // + producer warp
constexpr int kBarAll = 1;        // named barrier: all consumers
constexpr int kBarGroup = 2;      // named barriers 2, 3: consumer groups of 8 warps
constexpr int kMaxRing = 8;       // upper bound of ring stages (barrier arrays)
constexpr int kMaxChunksP2 = 2;   // 32-column chunks per consumer warp per gate/up stage (ks <= 1024)

__device__ __forceinline__ int fpad(int bytes) { return (bytes % 128 == 0) ? bytes + 64 : bytes; }

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(n) : "memory");
}

// Grid barrier, one thread per CTA.  ctr counts arrivals over the whole launch;
// barrier number `nb` (1-based) completes when ctr reaches nb * G.  Gives up
// when another CTA aborted or after kWaitNs.
__device__ bool grid_sync(const FusedParams &p, unsigned nb) {
  unsigned *ctr = p.ws.sync, *gabort = p.ws.sync + 2;
  red_release_add(ctr, 1u);
  const unsigned target = nb * gridDim.x;
  const unsigned long long t0 = global_ns();
  // one load per poll, so the count is seen within one L2 round trip of the
  // last arrival; the abort flag and the clock are read every 16th poll
  for (unsigned it = 1; ld_acquire(ctr) < target; ++it) {
    if ((it & 15u) == 0) {
      if (ld_relaxed(gabort)) return false;
      if (global_ns() - t0 > kWaitNs) {
        atomicOr(p.ws.err, DFV_DEVERR_GRID_WAIT);
        atomicExch(gabort, 1u);
        return false;
      }
    }
  }
  return true;
}

// The router rows of this CTA's experts b, b+G, ... start towards L2.  They are
// weights no kernel writes, so this may run before griddepcontrol.wait, while
// the previous launch drains; nothing else does.
__device__ __forceinline__ void prefetch_router_rows(const FusedParams &p) {
  const int e = blockIdx.x + (int)threadIdx.x * gridDim.x;
  if (threadIdx.x < 8 && e < p.E)
    prefetch_l2(reinterpret_cast<const char *>(p.wr) + (size_t)e * p.d * 2, (uint32_t)p.d * 2);
}

__device__ __forceinline__ void load8_bf16(const void *base, size_t elem, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(base) + elem);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ float rnd_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Routing tables in the calling CTA's shared memory.
// With a shared expert (p.ns = 1) the tables go on past the routed pairs: pair
// k*K + t is row t's shared slot (expert E, weight 1), and E is the last woken
// expert.
struct RouteSmem {
  int *idx;        // [k*K + ns*k]  expert of pair t*K+s, by descending logit
  float *w;        // [k*K + ns*k]  routing weight of the pair
  int *woken;      // [E + ns]      ascending ids of the woken experts
  int *off;        // [E + ns + 1]  per woken expert: first position in the sorted pair list
  int *eoff;       // [E]           per routed expert id: first position in the sorted pair list
  int *gat;        // [k*K + ns*k]  pair ids sorted by (expert, token)
  unsigned *mask;  // [kMaxBlock * E/32] experts chosen by each row
  float *inv;      // [kMaxBlock] 1/rms of each row (fuse_norm)
  int *wsum, *csum;  // [kFW] scan scratch
  int *nw;         // woken count
  volatile int *abort;
  volatile int *bad;  // set when the tables fail their check (zeroed by the caller)
};

// P0 + grid barrier 1 + P1, run by the kFW consumer warps of every CTA (named
// barrier kBarAll over kFC threads).
//   P0  router GEMV (optionally on RMSNorm(x) rounded to bf16): CTA b computes
//       the logits of experts b, b+G, ...; each (token, expert) dot product is
//       one warp's, in a fixed order, so a token's logit depends on nothing but
//       its own row.
//   P1  every CTA derives the whole routing decision itself from the logits:
//       top-K per row (warp per row, redux max/min: largest logit, lowest id
//       among equals), routing weights, woken union, per-expert pair offsets
//       (block scan) and the (expert, token)-sorted pair list, then appends
//       the shared expert (when p.ns).  CTA 0 also publishes the decision to
//       the workspace and the routed part to the caller's copies.
// `between` runs on the same threads after P0 and before grid barrier 1 (work
// that needs neither the other CTAs' logits nor the routing decision).
template <class Between>
__device__ __forceinline__ void fused_route(const FusedParams &p, const RouteSmem &r, Between &&between) {
  const int k = p.k, d = p.d, E = p.E, K = p.K;
  const int G = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // lane l takes the 16-byte pieces l, l+32, ... of a row, 8 at a time with
  // all their loads in flight; the sums run in piece order
  const int cpr = d / 8;
  if (p.fuse_norm) {
    if (warp < k) {
      const int t = warp;
      const uint16_t *xr = reinterpret_cast<const uint16_t *>(p.x) + (size_t)t * d;
      float ss = 0.f;
      for (int c0 = 0; c0 < cpr; c0 += 256) {
        uint4 xv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          xv[i] = c < cpr ? *reinterpret_cast<const uint4 *>(xr + (size_t)c * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + lane + 32 * i < cpr) {
            const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float a = bf16_lo(w4[h]), b = bf16_hi(w4[h]);
              ss = fmaf(a, a, ss);
              ss = fmaf(b, b, ss);
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) r.inv[t] = 1.0f / sqrtf(ss / (float)d + p.eps);
    }
    bar_sync_n(kBarAll, kFC);
  }
  // the (token, expert) dot products of this CTA's experts b, b+G, ... spread
  // over all warps: pair q = slot * k + t on warp q mod 16 (each dot product is
  // computed the same way whichever warp takes it)
  {
    const int n_e = blockIdx.x < E ? (E - 1 - blockIdx.x) / G + 1 : 0;
    for (int q = warp; q < n_e * k; q += kFW) {
      const int t = q % k, e = blockIdx.x + (q / k) * G;
      const uint16_t *xr = reinterpret_cast<const uint16_t *>(p.x) + (size_t)t * d;
      const float inv = p.fuse_norm ? r.inv[t] : 1.f;
      const uint16_t *wr = reinterpret_cast<const uint16_t *>(p.wr) + (size_t)e * d;
      float acc = 0.f;
      for (int c0 = 0; c0 < cpr; c0 += 256) {
        uint4 xv[8], wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          xv[i] = wv[i] = make_uint4(0u, 0u, 0u, 0u);
          if (c < cpr) {
            xv[i] = *reinterpret_cast<const uint4 *>(xr + (size_t)c * 8);
            wv[i] = *reinterpret_cast<const uint4 *>(wr + (size_t)c * 8);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + lane + 32 * i < cpr) {
            const uint32_t x4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            const uint32_t w4[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float a = bf16_lo(x4[h]), b = bf16_hi(x4[h]);
              if (p.fuse_norm) {
                a = rnd_bf16(a * inv);
                b = rnd_bf16(b * inv);
              }
              acc = fmaf(a, bf16_lo(w4[h]), acc);
              acc = fmaf(b, bf16_hi(w4[h]), acc);
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) p.ws.logits[(size_t)t * E + e] = acc;
    }
  }
  for (int i = tid; i < kMaxBlock * (kMaxExperts / 32); i += kFC) r.mask[i] = 0u;
  between();
  bar_sync_n(kBarAll, kFC);
  // ---- grid barrier 1: every CTA's logits are published
  if (tid == 0 && !grid_sync(p, 1)) *r.abort = 1;
  bar_sync_n(kBarAll, kFC);

  // ---------------------------------------------------------------- P1: routing
  // Warp t: top-K of row t (lane holds experts lane + 32 q), then the routing
  // weights in parallel over the K lanes.
  if (warp < k) {
    const int t = warp;
    uint32_t key[8];
    float val[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      val[q] = (e < E) ? __ldcg(p.ws.logits + (size_t)t * E + e) : 0.f;
      key[q] = (e < E) ? max(float_key(val[q]), 1u) : 0u;
    }
    int sel_id = 0;
    float sel_val = 0.f;
    for (int s = 0; s < K; ++s) {
      uint32_t bk = 0;
      int bq = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (key[q] > bk) { bk = key[q]; bq = q; }
      float bv = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q == bq) bv = val[q];
      const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t cand = (bk == m) ? (uint32_t)(lane + 32 * bq) : 0xffffffffu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      const float wv = __shfl_sync(0xffffffffu, bv, (int)(win & 31));
      if ((int)(win & 31) == lane) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q == (int)(win >> 5)) key[q] = 0u;
      }
      if (lane == s) { sel_id = (int)win; sel_val = wv; }
    }
    const float m0 = __shfl_sync(0xffffffffu, sel_val, 0);
    const float z = (lane < K) ? expf(sel_val - m0) : 0.f;
    float den = 0.f;
    if (p.norm_topk) {
      den = z;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (lane + 32 * q < E) den += expf(val[q] - m0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane < K) {
      r.idx[t * K + lane] = sel_id;
      r.w[t * K + lane] = z / den;
      atomicOr(&r.mask[t * (kMaxExperts / 32) + (sel_id >> 5)], 1u << (sel_id & 31));
    }
  }
  bar_sync_n(kBarAll, kFC);
  // per-expert pair counts from the row masks
  if (tid < E) {
    int cnt = 0;
    for (int t = 0; t < k; ++t) cnt += (r.mask[t * (kMaxExperts / 32) + (tid >> 5)] >> (tid & 31)) & 1u;
    r.eoff[tid] = cnt;
  }
  bar_sync_n(kBarAll, kFC);
  {
    // exclusive scans over experts (E <= 256 <= 8 warps of threads)
    int flag = 0, cnt = 0;
    if (tid < E) { cnt = r.eoff[tid]; flag = cnt > 0; }
    int fi = flag, ci = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, fi, o), b = __shfl_up_sync(0xffffffffu, ci, o);
      if (lane >= o) { fi += a; ci += b; }
    }
    if (lane == 31) { r.wsum[warp] = fi; r.csum[warp] = ci; }
    bar_sync_n(kBarAll, kFC);
    int wb = 0, cb = 0, nW = 0;
    for (int w = 0; w < kFW; ++w) {
      if (w < warp) { wb += r.wsum[w]; cb += r.csum[w]; }
      nW += r.wsum[w];
    }
    const int wpos = wb + fi - flag, off = cb + ci - cnt;
    if (tid < E) r.eoff[tid] = off;
    if (flag) { r.woken[wpos] = tid; r.off[wpos] = off; }
    if (tid == 0) { r.off[nW] = k * K; *r.nw = nW; }
  }
  bar_sync_n(kBarAll, kFC);
  for (int q = tid; q < k * K; q += kFC) {
    const int t = q / K, ex = r.idx[q];
    int rank = 0;
    for (int t2 = 0; t2 < t; ++t2) rank += (r.mask[t2 * (kMaxExperts / 32) + (ex >> 5)] >> (ex & 31)) & 1u;
    r.gat[r.eoff[ex] + rank] = q;
  }
  const int ns = p.ns ? 1 : 0, nP = k * K + ns * k, nE = E + ns;  // pairs, expert ids
  if (ns) {
    // the shared expert: the last woken expert (id E, above every routed id),
    // selected by every row with weight 1
    if (tid == 0) {
      const int nW = *r.nw;
      r.woken[nW] = E;
      r.off[nW + 1] = nP;
      *r.nw = nW + 1;
    }
    if (tid < k) {
      r.idx[k * K + tid] = E;
      r.w[k * K + tid] = 1.f;
      r.gat[k * K + tid] = k * K + tid;
    }
  }
  bar_sync_n(kBarAll, kFC);
  // every index the later phases take from these tables is checked once here:
  // woken ids ascending and < E + ns, offsets rising by 1..k and ending at
  // the pair count, and every sorted pair id below it, filed under the expert
  // it chose
  {
    const int nW = *r.nw;
    bool bad = tid == 0 && (nW < 1 || nW > nE || nW > k * K + ns || r.off[0] != 0 || r.off[nW] != nP);
    if (!bad && tid < nW && nW <= nE) {
      const int e = r.woken[tid], m = r.off[tid + 1] - r.off[tid];
      bad = e < 0 || e >= nE || (tid > 0 && e <= r.woken[tid - 1]) || m < 1 || m > k;
    }
    if (!bad && tid < nP && nW >= 1 && nW <= nE) {
      const int q = r.gat[tid];
      // the expert whose pair range holds position tid
      int lo = 0, hi = nW - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (r.off[mid] <= tid) lo = mid; else hi = mid - 1;
      }
      bad = q < 0 || q >= nP || r.idx[q] != r.woken[lo];
    }
    if (bad) *r.bad = 1;
  }
  bar_sync_n(kBarAll, kFC);
  if (*r.bad) {
    if (tid == 0) atomicOr(p.ws.err, DFV_DEVERR_ROUTING);
    *r.abort = 1;
  }
  if (blockIdx.x == 0) {
    const int nW = *r.nw;
    for (int q = tid; q < k * K; q += kFC) {
      p.ws.topk_idx[q] = r.idx[q];
      if (p.u_idx) p.u_idx[q] = r.idx[q];
    }
    for (int q = tid; q < nP; q += kFC) {
      p.ws.topk_w[q] = r.w[q];
      p.ws.gather[q] = r.gat[q];
    }
    for (int i = tid; i < nW; i += kFC) { p.ws.woken[i] = r.woken[i]; p.ws.offsets[i] = r.off[i]; }
    if (tid == 0) {
      p.ws.offsets[nW] = r.off[nW];
      *p.ws.n_woken = nW;
      if (p.u_nw) *p.u_nw = nW - ns;  // the caller's count: routed experts only
    }
  }
}

}  // namespace
}  // namespace dfv
