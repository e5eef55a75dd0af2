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
constexpr int kBarProducer = 7;   // named barrier: warp 0 releases the producer (64 threads)
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
__device__ __forceinline__ void prefetch_router_rows(const void *wr, int E, int d) {
  const int e = blockIdx.x + (int)threadIdx.x * gridDim.x;
  if (threadIdx.x < 8 && e < E) prefetch_l2(reinterpret_cast<const char *>(wr) + (size_t)e * d * 2, (uint32_t)d * 2);
}
__device__ __forceinline__ void prefetch_router_rows(const FusedParams &p) { prefetch_router_rows(p.wr, p.E, p.d); }

// Arrive on named barrier `id` (n threads in all) without waiting.
__device__ __forceinline__ void bar_arrive_n(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Start fetching a tensor map (kernel parameter, generic address) into the
// descriptor cache before its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
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
  unsigned *tmask; // [E]           bit t set when row t selected the expert
  float *inv;      // [kMaxBlock] 1/rms of each row (fuse_norm)
  int *nw;         // woken count
  volatile int *abort;
  volatile int *bad;  // set when the tables fail their check (zeroed by the caller)
};

// What the routing prologue needs, copied out of the kernel parameters and
// passed by value to the non-inlined prologue functions, so that they keep
// every field in registers (through a reference the compiler would reload
// them after each store it cannot prove distinct).
struct RouteArgs {
  int k, d, E, K, fuse_norm, norm_topk, ns;
  unsigned gb;              // grid barriers the launch completed before this layer
  float eps;
  const uint16_t *wr;       // router [E][d] bf16
  const uint16_t *xs;       // x rows [k][d] bf16 (shared memory, or p.x)
  uint32_t xbar;            // mbarrier of the x copy (0: xs is p.x)
  float *logits;            // workspace logits [k][E]
  unsigned *err, *sync;     // workspace error word, grid-barrier words
  int32_t *topk_idx, *woken, *offsets, *gather, *n_woken;  // workspace copies (CTA 0)
  float *topk_w;
  int32_t *u_idx, *u_nw;    // the caller's copies (CTA 0)
  // shared-memory tables
  int *idx;        // [k*K + ns*k]  expert of pair t*K+s, by descending logit
  float *w;        // [k*K + ns*k]  routing weight of the pair
  int *s_woken;    // [E + ns]      ascending ids of the woken experts
  int *off;        // [E + ns + 1]  per woken expert: first position in the sorted pair list
  int *eoff;       // [E]           per routed expert id: first position in the sorted pair list
  int *gat;        // [k*K + ns*k]  pair ids sorted by (expert, token)
  unsigned *tmask; // [E]           bit t set when row t selected the expert
  float *inv;      // [kMaxBlock]   1/rms of each row (fuse_norm)
  int *nw;         // woken count
  volatile int *abort;
  volatile int *bad;  // set when the tables fail their check (zeroed by the caller)
};

__device__ __forceinline__ RouteArgs route_args(const FusedParams &p, const RouteSmem &r, const uint16_t *xs,
                                                uint32_t xbar) {
  RouteArgs a;
  a.k = p.k; a.d = p.d; a.E = p.E; a.K = p.K;
  a.fuse_norm = p.fuse_norm; a.norm_topk = p.norm_topk; a.ns = p.ns ? 1 : 0;
  a.gb = 0;
  a.eps = p.eps;
  a.wr = reinterpret_cast<const uint16_t *>(p.wr);
  a.xs = xs;
  a.xbar = xbar;
  a.logits = p.ws.logits;
  a.err = p.ws.err;
  a.sync = p.ws.sync;
  a.topk_idx = p.ws.topk_idx; a.woken = p.ws.woken; a.offsets = p.ws.offsets; a.gather = p.ws.gather;
  a.n_woken = p.ws.n_woken; a.topk_w = p.ws.topk_w;
  a.u_idx = p.u_idx; a.u_nw = p.u_nw;
  a.idx = r.idx; a.w = r.w; a.s_woken = r.woken; a.off = r.off; a.eoff = r.eoff; a.gat = r.gat;
  a.tmask = r.tmask; a.inv = r.inv; a.nw = r.nw; a.abort = r.abort; a.bad = r.bad;
  return a;
}

// grid_sync on the raw workspace words (for the non-inlined prologue).
__device__ __forceinline__ bool grid_sync_raw(unsigned *sync, unsigned *err, unsigned nb) {
  unsigned *ctr = sync, *gabort = sync + 2;
  red_release_add(ctr, 1u);
  const unsigned target = nb * gridDim.x;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1; ld_acquire(ctr) < target; ++it) {
    if ((it & 15u) == 0) {
      if (ld_relaxed(gabort)) return false;
      if (global_ns() - t0 > kWaitNs) {
        atomicOr(err, DFV_DEVERR_GRID_WAIT);
        atomicExch(gabort, 1u);
        return false;
      }
    }
  }
  return true;
}

// The k rows of x start towards shared memory (one bulk copy per row, all on
// mbarrier `xbar`), issued by one thread after griddepcontrol.wait: x is the
// previous launch's output in a stack.  `dst` must hold k * d bf16 and be
// 16-byte aligned; d * 2 is a multiple of 16.
__device__ __forceinline__ void stage_x_rows(const FusedParams &p, uint32_t dst, uint32_t xbar) {
  const uint32_t rb = (uint32_t)p.d * 2;
  mbar_expect_tx(xbar, rb * (uint32_t)p.k);
  for (int t = 0; t < p.k; ++t)
    bulk_g2s(dst + (uint32_t)t * rb, reinterpret_cast<const uint16_t *>(p.x) + (size_t)t * p.d, rb, xbar);
}

// P0, run by the kFW consumer warps of every CTA (named barrier kBarAll over
// kFC threads).  Router GEMV, optionally on RMSNorm(x) rounded to bf16: CTA b
// computes the logits of experts b, b+G, ....  r.xs holds the k rows of x
// (bf16, row stride d), in shared memory once r.xbar completes (xbar == 0:
// xs is p.x in global memory).  The CTA's n_e experts share its warps: kFW /
// n_e warps per expert, each loading its expert's router row once (issued
// before the wait for x, so the two transfers overlap) and taking every
// (kFW / n_e)-th token.  Each (token, expert) dot product is one warp's,
// computed in one fixed order whichever warp takes it, so a token's logit
// depends on nothing but its own row.
__device__ __forceinline__ void route_p0(const RouteArgs &r) {
  const int k = r.k, d = r.d, E = r.E;
  const int G = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t *xs = r.xs;
  for (int i = tid; i < kMaxExperts; i += kFC) r.tmask[i] = 0u;
  const int cpr = d / 8;  // 16-byte pieces per row; lane l takes pieces l, l+32, ...
  const int n_e = blockIdx.x < E ? (E - 1 - blockIdx.x) / G + 1 : 0;
  const int wpe = n_e >= kFW ? 1 : (n_e > 0 ? kFW / n_e : kFW);  // warps per expert
  const int jstep = kFW / wpe;
  const int j0 = warp / wpe;
  const bool active = n_e > 0 && j0 < n_e && warp < wpe * jstep;
  // the first 256 pieces of this warp's first router row, in flight while x arrives
  uint4 wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    wv[i] = (active && c < cpr)
                ? __ldg(reinterpret_cast<const uint4 *>(r.wr + (size_t)(blockIdx.x + j0 * G) * d + (size_t)c * 8))
                : make_uint4(0u, 0u, 0u, 0u);
  }
  if (r.xbar) {
    // one thread waits (bounded) for the x copy; the named barrier then
    // orders the copied rows before every consumer's reads, and all consumers
    // see the same abort flag after it
    if (tid == 0 && !mbar_wait(r.xbar, 0u, r.err, DFV_DEVERR_STAGE_WAIT, r.abort)) *r.abort = 1;
    bar_sync_n(kBarAll, kFC);
    if (*r.abort) return;
  }
  if (r.fuse_norm) {
    if (warp < k) {
      const uint16_t *xr = xs + (size_t)warp * d;
      float ss = 0.f;
      for (int c = lane; c < cpr; c += 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xr + (size_t)c * 8);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float a = bf16_lo(w4[h]), b = bf16_hi(w4[h]);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) r.inv[warp] = 1.0f / sqrtf(ss / (float)d + r.eps);
    }
    bar_sync_n(kBarAll, kFC);
  }
  if (!active) return;
  // rolled loops over experts, tokens and 256-piece chunks of a row: this code
  // runs once per launch, so its size (cold instruction fetch) counts more
  // than its loop overhead
  int cur_j = j0, cur_c0 = 0;  // the router-row chunk wv holds
#pragma unroll 1
  for (int j = j0; j < n_e; j += jstep) {
    const int e = blockIdx.x + j * G;
    const uint16_t *wr = r.wr + (size_t)e * d;
#pragma unroll 1
    for (int t = warp % wpe; t < k; t += wpe) {
      const uint16_t *xr = xs + (size_t)t * d;
      const float inv = r.fuse_norm ? r.inv[t] : 1.f;
      float acc = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < cpr; c0 += 256) {
        if (cur_j != j || cur_c0 != c0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + lane + 32 * i;
            wv[i] = c < cpr ? __ldg(reinterpret_cast<const uint4 *>(wr + (size_t)c * 8)) : make_uint4(0u, 0u, 0u, 0u);
          }
          cur_j = j;
          cur_c0 = c0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < cpr) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xr + (size_t)c * 8);
            const uint32_t x4[4] = {xv.x, xv.y, xv.z, xv.w};
            const uint32_t w4[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float a = bf16_lo(x4[h]), b = bf16_hi(x4[h]);
              if (r.fuse_norm) {
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
      if (lane == 0) r.logits[(size_t)t * E + e] = acc;
    }
  }
}

// Top-K of logit row t, by one warp (lane l holds experts l + 32 q): largest
// logit first, lowest id among equals; then the routing weights.  Returns, in
// lane s < K, the s-th selected expert; its weight is z / den.
__device__ __forceinline__ void route_row(const RouteArgs &r, int t, int lane, int &sel_id, float &z, float &den) {
  const int E = r.E, K = r.K;
  uint32_t key[8];
  float val[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    val[q] = (e < E) ? __ldcg(r.logits + (size_t)t * E + e) : 0.f;
    key[q] = (e < E) ? max(float_key(val[q]), 1u) : 0u;
  }
  sel_id = 0;
  float sel_val = 0.f;
  for (int s = 0; s < K; ++s) {
    // every lane rescans its eight keys each round (no divergent update)
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
  z = (lane < K) ? expf(sel_val - m0) : 0.f;
  den = 0.f;
  if (r.norm_topk) {
    den = z;
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (lane + 32 * q < E) den += expf(val[q] - m0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
}

// Writes the routing decision in the calling CTA's tables to the workspace
// (CTA 0) and the routed part to the caller's copies.
__device__ __forceinline__ void route_publish(const RouteArgs &r) {
  const int k = r.k, K = r.K, tid = threadIdx.x;
  const int nP = k * K + r.ns * k;
  if (blockIdx.x == 0) {
    const int nW = *r.nw;
    for (int q = tid; q < k * K; q += kFC) {
      r.topk_idx[q] = r.idx[q];
      if (r.u_idx) r.u_idx[q] = r.idx[q];
    }
    for (int q = tid; q < nP; q += kFC) {
      r.topk_w[q] = r.w[q];
      r.gather[q] = r.gat[q];
    }
    for (int i = tid; i < nW; i += kFC) { r.woken[i] = r.s_woken[i]; r.offsets[i] = r.off[i]; }
    if (tid == 0) {
      r.offsets[nW] = r.off[nW];
      *r.n_woken = nW;
      if (r.u_nw) *r.u_nw = nW - r.ns;  // the caller's count: routed experts only
    }
  }
}

// P1 of a single-token block (k = 1), by warp 0 alone: its K experts are the
// woken ones, one pair each, so the tables are the selection sorted by id
// (each selected expert's rank among the K is its woken position, its pair
// position and its offset).  The same tables as the general path builds,
// without the per-expert masks, the scan and their block barriers.
template <class AfterScan>
__device__ __forceinline__ void route_p1_single(const RouteArgs &r, AfterScan &&after_scan) {
  const int E = r.E, K = r.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp == 0) {
    int sel_id;
    float z, den;
    route_row(r, 0, lane, sel_id, z, den);
    int rank = 0;  // selected ids are distinct: the rank is the woken position
    for (int j = 0; j < K; ++j) rank += (__shfl_sync(0xffffffffu, sel_id, j) < sel_id) ? 1 : 0;
    const bool in = lane < K;
    const unsigned seen = __reduce_or_sync(0xffffffffu, in ? 1u << rank : 0u);
    const bool bad = __any_sync(0xffffffffu, in && (sel_id < 0 || sel_id >= E)) || seen != (1u << K) - 1u;
    if (in) {
      r.idx[lane] = sel_id;
      r.w[lane] = z / den;
      r.s_woken[rank] = sel_id;
      r.off[rank] = rank;
      r.gat[rank] = lane;  // pair t * K + s of row 0 is s
    }
    if (lane == 0) {
      int nW = K;
      r.off[K] = K;
      if (r.ns) {
        // the shared expert: the last woken expert, selected by row 0 with weight 1
        r.s_woken[K] = E;
        r.off[K + 1] = K + 1;
        r.idx[K] = E;
        r.w[K] = 1.f;
        r.gat[K] = K;
        ++nW;
      }
      if (bad) {
        *r.bad = 1;
        atomicOr(r.err, DFV_DEVERR_ROUTING);
        *r.abort = 1;
      }
      *r.nw = *r.abort ? 0 : nW;
    }
    __syncwarp();
    if (lane == 0) after_scan(1);  // every routed expert took the one row
    __syncwarp();
    bar_arrive_n(kBarProducer, 64);
  }
  bar_sync_n(kBarAll, kFC);
  route_publish(r);
}

// grid barrier 1 + P1, run by the kFW consumer warps of every CTA.  Every CTA
// derives the whole routing decision itself from the published logits:
// top-K per row (warp per row, route_row), per-expert token masks, woken
// union and pair offsets (one warp's scan over the experts), the (expert,
// token)-sorted pair list (a pair's position is its expert's offset plus the
// number of earlier rows that chose the expert), then the shared expert (when
// p.ns).  Lane 0 of warp 0 calls after_scan(most rows any routed expert took)
// as soon as the woken list and the offsets are in shared memory.  The tables
// are checked before anything indexes with them.  CTA 0 also publishes the
// decision to the workspace and the routed part to the caller's copies.
// SINGLE (a kernel instantiated for single-token blocks only, k = 1) takes
// route_p1_single instead; the other instantiations do not carry that code.
template <bool SINGLE, class AfterScan>
__device__ __forceinline__ void route_p1(const RouteArgs &r, AfterScan &&after_scan) {
  const int k = r.k, E = r.E, K = r.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- grid barrier 1: every CTA's logits are published
  bar_sync_n(kBarAll, kFC);
  if (tid == 0 && !grid_sync_raw(r.sync, r.err, r.gb + 1)) *r.abort = 1;
  bar_sync_n(kBarAll, kFC);
  if constexpr (SINGLE) {
    route_p1_single(r, after_scan);
    return;
  }

  // Warp t: top-K of row t, then the per-expert token masks.
  if (warp < k) {
    const int t = warp;
    int sel_id;
    float z, den;
    route_row(r, t, lane, sel_id, z, den);
    if (lane < K) {
      r.idx[t * K + lane] = sel_id;
      r.w[t * K + lane] = z / den;
      atomicOr(&r.tmask[sel_id], 1u << t);
    }
  }
  bar_sync_n(kBarAll, kFC);
  // woken union and pair offsets: warp 0, lane l holding experts 8l .. 8l+7
  // (E <= 256); exclusive scans of the woken flags and the pair counts
  if (warp == 0) {
    int cnt[8], nf = 0, nc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      cnt[i] = e < E ? __popc(r.tmask[e]) : 0;
      nf += cnt[i] > 0;
      nc += cnt[i];
    }
    int cmax = 0;  // most rows any routed expert took
#pragma unroll
    for (int i = 0; i < 8; ++i) cmax = max(cmax, cnt[i]);
    cmax = (int)__reduce_max_sync(0xffffffffu, (unsigned)cmax);
    int fi = nf, ci = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, fi, o), b = __shfl_up_sync(0xffffffffu, ci, o);
      if (lane >= o) { fi += a; ci += b; }
    }
    int wpos = fi - nf, off = ci - nc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        r.eoff[e] = off;
        if (cnt[i] > 0) { r.s_woken[wpos] = e; r.off[wpos] = off; ++wpos; }
        off += cnt[i];
      }
    }
    if (lane == 31) {
      r.off[fi] = k * K;
      int nW = fi;
      if (r.ns) {
        // the shared expert: the last woken expert (id E, above every routed
        // id), selected by every row with weight 1
        r.s_woken[nW] = E;
        r.off[nW + 1] = k * K + k;
        ++nW;
      }
      *r.nw = *r.abort ? 0 : nW;  // a CTA that gave up at the grid barrier takes no units
    }
    __syncwarp();
    if (lane == 0) after_scan(cmax);
    __syncwarp();
    // the woken list and the offsets are all the producer needs: release it
    bar_arrive_n(kBarProducer, 64);
  }
  bar_sync_n(kBarAll, kFC);
  for (int q = tid; q < k * K; q += kFC) {
    const int t = q / K, ex = r.idx[q];
    r.gat[r.eoff[ex] + __popc(r.tmask[ex] & ((1u << t) - 1u))] = q;
  }
  const int ns = r.ns, nP = k * K + ns * k, nE = E + ns;  // pairs, expert ids
  if (ns) {
    // the shared expert's pairs k*K + t, weight 1, in token order
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
      const int e = r.s_woken[tid], m = r.off[tid + 1] - r.off[tid];
      bad = e < 0 || e >= nE || (tid > 0 && e <= r.s_woken[tid - 1]) || m < 1 || m > k;
    }
    if (!bad && tid < nP && nW >= 1 && nW <= nE) {
      const int q = r.gat[tid];
      // the expert whose pair range holds position tid
      int lo = 0, hi = nW - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (r.off[mid] <= tid) lo = mid; else hi = mid - 1;
      }
      bad = q < 0 || q >= nP || r.idx[q] != r.s_woken[lo];
    }
    if (bad) *r.bad = 1;
  }
  bar_sync_n(kBarAll, kFC);
  if (*r.bad) {
    if (tid == 0) atomicOr(r.err, DFV_DEVERR_ROUTING);
    *r.abort = 1;
  }
  route_publish(r);
}

}  // namespace
}  // namespace dfv
