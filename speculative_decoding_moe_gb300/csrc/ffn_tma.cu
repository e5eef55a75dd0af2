// ffn_tma.cu -- TMA-staged grouped SwiGLU expert FFN and combine (bf16
// weights), one persistent CTA per SM.
//
// Same arithmetic as the register-direct kernels in ffn.cu ("Speculating on a
// Strix Halo", sections "What the pieces cost" and "The verify's own cost":
// tokens sorted by expert, one grouped launch per projection, the block's
// output the routing-weighted sum of each token's K experts), with the weight
// stream decoupled from the arithmetic:
//
//   * warp 8 is the producer: one thread walks the CTA's units and, for each
//     stage of a ring in shared memory, waits for the stage to be free, posts
//     the expected byte count on the stage's "full" mbarrier and issues the
//     copies: one 3-D tensor copy per gate/up matrix (its 8 rows) and per down
//     unit (its rs rows), as 128-byte segments with the 128-byte swizzle (1-D
//     bulk copies per row piece, into padded rows, when the maps cannot be
//     made);
//   * warps 0-7 consume: wait on "full", run the m16n8k16 MMAs from shared
//     memory, release the stage on its "empty" mbarrier, and do the per-unit
//     epilogues (cross-warp reduction, SwiGLU, weighted scatter) while the
//     producer keeps the next stages loading;
//   * a third launch combines: every output summed over its slots in slot
//     order (no per-unit ticket on the down kernel's path).
//
// h enters the down contraction rounded to bf16, as in the single-launch
// kernel.
//
// Every weight byte of a woken expert crosses HBM once.  In the swizzled
// stages MMA row g (and g + 8) reads stored row (g >> 1) | ((g & 1) << 2) (and
// that + 8), so the two rows of a quarter-warp's fragment loads are r and
// r + 4, whose 16-byte chunks the swizzle puts in opposite halves of the
// banks; the padded rows (a stride of 64 mod 128 bytes) get the same from the
// padding.  One copy per matrix and per down unit, instead of one per row
// piece, took the A3B layer at k = 16 from 201 to 181 us and the single-token
// layers 6-13% faster.  Every mbarrier wait
// is bounded (2 s); a timeout sets a bit in the workspace error word, the CTA
// stops, and the producer waits (bounded) for its copies in flight first.
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "dfv_internal.cuh"

namespace dfv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;
constexpr int kBarConsumers = 1;  // named barrier id for the consumer warps

__device__ __forceinline__ int pad_to_64mod128(int bytes) { return (bytes % 128 == 0) ? bytes + 64 : bytes; }

__device__ __forceinline__ void unit_range_tma(int U, int &lo, int &hi) {
  lo = (int)(((long long)blockIdx.x * U) / gridDim.x);
  hi = (int)(((long long)(blockIdx.x + 1) * U) / gridDim.x);
}

// Wait (bounded) until the copies of the last min(issued, S) stage fills have
// landed, so no bulk copy targets this CTA's shared memory after it exits.
__device__ void drain_stages(uint32_t full0, int issued, int S, unsigned *err) {
  volatile int never = 0;  // the drain ignores the CTA's abort flag
  for (int j = issued - S < 0 ? 0 : issued - S; j < issued; ++j)
    if (!mbar_wait(full0 + 8 * (j % S), (j / S) & 1, err, DFV_DEVERR_DRAIN_WAIT, &never)) return;
}

// ----------------------------------------------------------------------------
// gate/up.  Unit = (woken expert, 8 d_ff rows); stage = that unit's 8 gate and
// 8 up rows over `ks` columns (nslices stages per unit).  Where half the
// shared-memory budget holds two stages beside the staged x rows (d up to
// 2048, with 512-column slices at d = 2048), two CTAs share an SM: 18 warps
// instead of 9 hide the stage and fragment latencies (the A3B layer at k = 16
// went from 164.9 to 151.0 us, the OLMoE-like one from 150.5 to 138.7 us).
// Shared memory (1024-aligned): stages[S] | xs[NT*8][rsx] | red[8][NT][32][4]
// f32 | full[S] | empty[S]; a stage is gate then up, each [ks/64][8][128 B]
// swizzled (tma_mode 1), or [16][rsg] padded rows (tma_mode 0).
template <int NT>
__global__ void __launch_bounds__(kTmaThreads, 2) gateup_tma_kernel(const __grid_constant__ FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // the 128-byte swizzle repeats every 1024 bytes: stages start 1024-aligned
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int d = p.d, I = p.I, K = p.K, ks = p.ks, S = p.stages, nsl = p.nslices;
  const int rsg = pad_to_64mod128(ks * 2);
  const int rsx = pad_to_64mod128(d * 2);
  const uint32_t sbase = smem_u32(smem);
  // stage layout: padded rows (mode 0), or [ks/64][8 rows][128 B] segments
  // with the 128-byte swizzle (mode 1); up rows follow the gate rows
  const uint32_t stage_bytes = p.tma_mode ? 32u * ks : 16u * rsg;
  const uint32_t up_off = p.tma_mode ? 16u * ks : 8u * rsg;
  const uint32_t xbase = sbase + S * stage_bytes;
  float *red = reinterpret_cast<float *>(smem + S * stage_bytes + (size_t)NT * 8 * rsx);
  const uint32_t full0 = smem_u32(red + kConsumerWarps * NT * 32 * 4);
  const uint32_t empty0 = full0 + 8 * S;
  __shared__ int s_tok[16];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();

  const int nW = *p.ws.n_woken;
  const int tiles = I / kGateTile;
  int lo, hi;
  unit_range_tma(nW * tiles, lo, hi);

  if (warp == kConsumerWarps) {
    // ---------------- producer
    if (lane == 0) {
      const uint16_t *wg = reinterpret_cast<const uint16_t *>(p.wg);
      const uint16_t *wu = reinterpret_cast<const uint16_t *>(p.wu);
      const uint64_t pol = l2_evict_first();  // expert weights are read once per launch
      int it = 0;
      bool ok = true;
      for (int u = lo; u < hi && ok; ++u) {
        const int e = p.ws.woken[u / tiles], i0 = (u % tiles) * kGateTile;
        for (int sl = 0; sl < nsl; ++sl, ++it) {
          const int s = it % S;
          if (!mbar_wait(empty0 + 8 * s, ((it / S) & 1) ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * s, dst = sbase + s * stage_bytes;
          mbar_expect_tx(fb, 16u * ks * 2);
          if (p.tma_mode) {  // [ks/64][8 rows][128 B], swizzled: one box per matrix
            tma_3d_hint(dst, &p.tm_wg, 0, e * I + i0, sl * (ks / 64), fb, pol);
            tma_3d_hint(dst + up_off, &p.tm_wu, 0, e * I + i0, sl * (ks / 64), fb, pol);
          } else {  // one padded row piece per copy
            for (int r = 0; r < 8; ++r) {
              const size_t row = ((size_t)e * I + i0 + r) * d + (size_t)sl * ks;
              bulk_g2s(dst + r * rsg, wg + row, ks * 2, fb);
              bulk_g2s(dst + (8 + r) * rsg, wu + row, ks * 2, fb);
            }
          }
        }
      }
      drain_stages(full0, it, S, p.ws.err);
    }
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const uint32_t pr = (uint32_t)((g >> 1) | ((g & 1) << 2));  // stored row of MMA row g (mode 1)
  const int cps = ks / 32;  // 32-column chunks per slice
  const int c0 = warp * cps / kConsumerWarps, c1 = (warp + 1) * cps / kConsumerWarps;
  const uint16_t *xg = reinterpret_cast<const uint16_t *>(p.x);
  const int cpr = d / 8;
  int cur = -1, m = 0, off = 0, it = 0;
  bool dead = false;  // after a failed wait: keep the barrier schedule, skip the work
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, i0 = (u % tiles) * kGateTile;
    if (wi != cur) {
      bar_sync_n(kBarConsumers, kConsumers);
      cur = wi;
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      if (tid < m) s_tok[tid] = pair_token(p.ws.gather[off + tid], p.k, K);
      bar_sync_n(kBarConsumers, kConsumers);
      for (int idx = tid; idx < m * cpr; idx += kConsumers) {
        const int j = idx / cpr, q = idx % cpr;
        const uint4 v = *reinterpret_cast<const uint4 *>(xg + (size_t)s_tok[j] * d + q * 8);
        *reinterpret_cast<uint4 *>(smem + (xbase - sbase) + (size_t)j * rsx + q * 16) = v;
      }
      bar_sync_n(kBarConsumers, kConsumers);
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    for (int sl = 0; sl < nsl; ++sl, ++it) {
      const int s = it % S;
      if (!dead && !mbar_wait(full0 + 8 * s, (it / S) & 1, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) dead = true;
      if (dead) continue;
      const uint32_t st = sbase + s * stage_bytes;
      for (int ch = c0; ch < c1; ++ch) {
        // mode 1: MMA row g reads stored row pr (rows 0,4,1,5,...): the two rows
        // of a quarter-warp's loads then sit in opposite halves of the swizzle
        const uint32_t o = p.tma_mode ? (ch >> 1) * 1024u + pr * 128u + ((((ch & 1) * 4 + c) ^ pr) << 4)
                                      : g * rsg + (ch * 4 + c) * 16;
        const uint4 ag = lds128(st + o);
        const uint4 au = lds128(st + up_off + o);
        const uint32_t xq = (uint32_t)(sl * (ks / 8) + ch * 4 + c) * 16;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (nt * 8 < m) {
            const int row = nt * 8 + g;
            uint4 b = make_uint4(0u, 0u, 0u, 0u);
            if (row < m) b = lds128(xbase + row * rsx + xq);
            mma_bf16(acc[nt], ag.x, au.x, ag.y, au.y, b.x, b.y);
            mma_bf16(acc[nt], ag.z, au.z, ag.w, au.w, b.z, b.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4 *>(red + ((warp * NT + nt) * 32 + lane) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    bar_sync_n(kBarConsumers, kConsumers);
    if (tid < NT * 64) {
      const int nt = tid >> 6, ln = (tid >> 1) & 31, q = tid & 1;
      const int tok = nt * 8 + 2 * (ln & 3) + q;
      if (tok < m) {
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) {
          gs += red[((w * NT + nt) * 32 + ln) * 4 + q];
          us += red[((w * NT + nt) * 32 + ln) * 4 + q + 2];
        }
        const int gr = ln >> 2;  // MMA row; mode 1 stores it as row (gr >> 1) | ((gr & 1) << 2)
        p.ws.h[(size_t)(off + tok) * I + i0 + (p.tma_mode ? ((gr >> 1) | ((gr & 1) << 2)) : gr)] = silu(gs) * us;
      }
    }
    bar_sync_n(kBarConsumers, kConsumers);
  }
}

// ----------------------------------------------------------------------------
// down.  Unit = (woken expert, rs rows of d); stage = those rows over the full
// d_ff.  Consumers: 2 row-tiles of 16 x 4 k-quarters (rs = 32) or 1 x 8
// (rs = 16).  Where half the shared-memory budget holds two 16-row stages
// (d_ff up to 1024), two CTAs share an SM: 18 warps instead of 9 hide the
// stage and L2 latencies (the A3B layer at k = 16 went from 180.8 to 167.7
// us, the OLMoE-like one from 162.0 to 153.0 us).  Wider d_ff (a multiple of
// 128) keeps two CTAs per SM with DS = 2 stages per unit, each holding half of
// d_ff (Qwen1.5-MoE-like layer 145.5 -> 134.7 us, Qwen3-235B-like 597.4 ->
// 552.9 us); each warp then takes an eighth of every half.  h of the expert's tokens is staged in bf16; w[t,s] * y goes to
// ys[pair], and the combine launch sums it.
// Shared memory (1024-aligned): stages[S] | h[NT*8][rsh] | red[8][NT][32][4]
// f32 | full[S] | empty[S]; a stage is [d_ff/64][rs][128 B] swizzled
// (tma_mode 1) or [rs][rsd] padded rows (tma_mode 0).
template <int NT, int DS>
__global__ void __launch_bounds__(kTmaThreads, 2) down_tma_kernel(const __grid_constant__ FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int d = p.d, I = p.I, S = p.stages, RS = p.rs;
  const int Ih = I / DS;  // d_ff columns per stage
  const int rsd = pad_to_64mod128(Ih * 2);
  const int rsh = pad_to_64mod128(I * 2);
  const uint32_t sbase = smem_u32(smem);
  // stage layout: padded rows (tma_mode 0), or [Ih/64][RS rows][128 B] with the
  // 128-byte swizzle from one tensor copy (tma_mode 1); a unit takes DS stages
  const uint32_t stage_bytes = p.tma_mode ? (uint32_t)RS * Ih * 2 : (uint32_t)RS * rsd;
  const uint32_t hhb = sbase + S * stage_bytes;
  float *red = reinterpret_cast<float *>(smem + S * stage_bytes + (size_t)NT * 8 * rsh);
  const uint32_t full0 = smem_u32(red + kConsumerWarps * NT * 32 * 4);
  const uint32_t empty0 = full0 + 8 * S;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();

  const int nW = *p.ws.n_woken;
  const int tiles = (d + RS - 1) / RS;
  int lo, hi;
  unit_range_tma(nW * tiles, lo, hi);

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const uint16_t *wd = reinterpret_cast<const uint16_t *>(p.wd);
      const uint64_t pol = l2_evict_first();  // expert weights are read once per launch
      int it = 0;
      bool ok = true;
      for (int u = lo; u < hi && ok; ++u) {
        const int e = p.ws.woken[u / tiles], r0 = (u % tiles) * RS;
        const int rows = min(RS, d - r0);
        for (int sl = 0; sl < DS; ++sl, ++it) {
          const int s = it % S;
          if (!mbar_wait(empty0 + 8 * s, ((it / S) & 1) ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * s, dst = sbase + s * stage_bytes;
          if (p.tma_mode) {  // one box of RS rows (rows past d are zero-filled and counted)
            mbar_expect_tx(fb, (uint32_t)RS * Ih * 2);
            tma_3d_hint(dst, &p.tm_wd, 0, e * d + r0, sl * (Ih / 64), fb, pol);
          } else {
            mbar_expect_tx(fb, (uint32_t)rows * Ih * 2);
            for (int r = 0; r < rows; ++r)
              bulk_g2s(dst + r * rsd, wd + ((size_t)e * d + r0 + r) * I + (size_t)sl * Ih, Ih * 2, fb);
          }
        }
      }
      drain_stages(full0, it, S, p.ws.err);
    }
    return;
  }

  const int g = lane >> 2, c = lane & 3;
  // swizzled stages: MMA rows g and g + 8 of a row tile read stored rows pr and
  // 8 + pr (rows 0,4,1,5,...), so a quarter-warp's two rows sit in opposite
  // halves of the swizzle
  const uint32_t pr = (uint32_t)((g >> 1) | ((g & 1) << 2));
  const int rtiles = RS / 16;                   // row tiles per unit (2 or 1)
  const int kparts = kConsumerWarps / rtiles;   // k parts (4 or 8)
  const int rw = warp % rtiles, kq = warp / rtiles;
  const int Cs = Ih / 32;  // 32-column chunks per stage
  const int c0 = kq * Cs / kparts, c1 = (kq + 1) * Cs / kparts;
  const int cpr = I / 8;
  int cur = -1, m = 0, off = 0, it = 0;
  bool dead = false;  // after a failed wait: keep the barrier schedule, skip the work
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, dt = u % tiles, r0 = dt * RS;
    const int rows = min(RS, d - r0);
    if (wi != cur) {
      bar_sync_n(kBarConsumers, kConsumers);
      cur = wi;
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      for (int idx = tid; idx < m * cpr; idx += kConsumers) {
        const int j = idx / cpr, q = idx % cpr;
        const float4 *src = reinterpret_cast<const float4 *>(p.ws.h + (size_t)(off + j) * I + q * 8);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t h2[4];
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
          h2[q2] = (uint32_t)f32_to_bf16_bits(v[2 * q2]) | ((uint32_t)f32_to_bf16_bits(v[2 * q2 + 1]) << 16);
        *reinterpret_cast<uint4 *>(smem + (hhb - sbase) + (size_t)j * rsh + q * 16) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
      }
      bar_sync_n(kBarConsumers, kConsumers);
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    for (int sl = 0; sl < DS; ++sl, ++it) {
      const int s = it % S;
      if (!dead && !mbar_wait(full0 + 8 * s, (it / S) & 1, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) dead = true;
      const uint32_t st = sbase + s * stage_bytes;
      if (!dead && rw * 16 < rows) {
        for (int ch = c0; ch < c1; ++ch) {
          const uint32_t ql = (uint32_t)(ch * 4 + c);                  // 16-byte piece within the stage
          const uint32_t q16 = (uint32_t)((sl * Cs + ch) * 4 + c) * 16;  // and within the h row
          uint32_t o0, o1;
          if (p.tma_mode) {
            o0 = (ql >> 3) * (uint32_t)(RS * 128) + (rw * 16 + pr) * 128u + (((ql & 7u) ^ pr) << 4);
            o1 = o0 + 1024u;
          } else {
            o0 = (rw * 16 + g) * rsd + ql * 16;
            o1 = (rw * 16 + g + 8) * rsd + ql * 16;
          }
          const uint4 a0 = lds128(st + o0);
          const uint4 a1 = lds128(st + o1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt * 8 < m) {
              const int row = nt * 8 + g;
              uint4 bh = make_uint4(0u, 0u, 0u, 0u);
              if (row < m) bh = lds128(hhb + row * rsh + q16);
              mma_bf16(acc[nt], a0.x, a1.x, a0.y, a1.y, bh.x, bh.y);
              mma_bf16(acc[nt], a0.z, a1.z, a0.w, a1.w, bh.z, bh.w);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4 *>(red + ((warp * NT + nt) * 32 + lane) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    bar_sync_n(kBarConsumers, kConsumers);
    // y[row][tok] = sum over k parts (fixed order); weighted by the pair's routing weight
    for (int idx = tid; idx < rtiles * NT * 128; idx += kConsumers) {
      const int q4 = idx & 3, ln = (idx >> 2) & 31, nt = (idx >> 7) % NT, rt = idx / (128 * NT);
      const int gr = ln >> 2;
      const int row = r0 + rt * 16 + (p.tma_mode ? ((gr >> 1) | ((gr & 1) << 2)) : gr) + ((q4 & 2) ? 8 : 0);
      const int tok = nt * 8 + 2 * (ln & 3) + (q4 & 1);
      if (tok < m && row < d) {
        float y = 0.f;
        for (int kp = 0; kp < kparts; ++kp) y += red[(((kp * rtiles + rt) * NT + nt) * 32 + ln) * 4 + q4];
        const int pair = p.ws.gather[off + tok];
        p.ws.ys[(size_t)pair * d + row] = p.ws.topk_w[pair] * y;
      }
    }
    bar_sync_n(kBarConsumers, kConsumers);  // red is free for the next unit
  }
}

// out[t] = residual[t] + sum over slots s of ys[t*K+s] (slot order) + the
// shared slot, every (t, r) once, after the down launch wrote every ys row.
__global__ void __launch_bounds__(256) combine_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  const int n = p.k * p.d;
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nthr = gridDim.x * blockDim.x;
  for (int idx = tid; idx < n; idx += nthr) {
    const int t = idx / p.d, r = idx - t * p.d;
    float s = 0.f;
    for (int sl = 0; sl < p.K; ++sl) s += __ldcg(p.ws.ys + (size_t)(t * p.K + sl) * p.d + r);
    if (p.ns) s += __ldcg(p.ws.ys + (size_t)(p.k * p.K + t) * p.d + r);
    if (p.residual) s = load_act(p.residual, (size_t)t * p.d + r, p.act) + s;
    store_act(p.out, (size_t)t * p.d + r, p.act, s);
  }
}

// ----------------------------------------------------------------------------
// host side
namespace {
int pad_host(int bytes) { return (bytes % 128 == 0) ? bytes + 64 : bytes; }
constexpr size_t kSmemBudget = 220 * 1024;
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char *why, size_t why_len);

// The maps of the TMA-staged kernels, 128-byte rows with the 128-byte swizzle:
// gate and up viewed as [d/64][E*I rows][64 columns], box {64, 8, ks/64}; down
// as [d_ff/64][E*d rows][64 columns], box {64, rs, d_ff/64}; cached per
// (weights, shape).  Mode 0 when any of them cannot be encoded.
void ffn_tensor_maps(FfnParams *p, const dfv_moe_layer *L, int ks, int rs, int dsl) {
  struct Maps {
    int mode;
    CUtensorMap wg, wu, wd;
  };
  static std::mutex mu;
  static std::map<std::tuple<const void *, const void *, const void *, int, int, int, int, int, int>, Maps> cache;
  p->tma_mode = 0;
  const int d = L->d, I = L->d_ff, E = L->n_experts + (L->n_shared ? 1 : 0), kst = ks;
  if (d % 64 || ks % 64 || ks / 64 > 256) return;
  const auto key = std::make_tuple(L->w_gate, L->w_up, L->w_down, d, I, E, kst, rs, dsl);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      p->tma_mode = it->second.mode;
      p->tm_wg = it->second.wg;
      p->tm_wu = it->second.wu;
      p->tm_wd = it->second.wd;
      return;
    }
  }
  char why[128];
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, sizeof why);
  Maps m = {};
  if (fn) {
    auto enc = [&](CUtensorMap *map, const void *base) {
      const cuuint64_t dims[3] = {64, (cuuint64_t)E * I, (cuuint64_t)d / 64};
      const cuuint64_t strides[2] = {(cuuint64_t)d * 2, 128};
      const cuuint32_t box[3] = {64, 8, (cuuint32_t)kst / 64};
      const cuuint32_t es[3] = {1, 1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // the down rows: [d_ff/64][rs rows][64 columns], box {64, rs, d_ff/64/dsl}
    auto encd = [&](CUtensorMap *map, const void *base) {
      const cuuint64_t dims[3] = {64, (cuuint64_t)E * d, (cuuint64_t)I / 64};
      const cuuint64_t strides[2] = {(cuuint64_t)I * 2, 128};
      const cuuint32_t box[3] = {64, (cuuint32_t)rs, (cuuint32_t)(I / 64 / dsl)};
      const cuuint32_t es[3] = {1, 1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (I % (64 * dsl) == 0 && I / 64 <= 256 && enc(&m.wg, L->w_gate) && enc(&m.wu, L->w_up) &&
        encd(&m.wd, L->w_down))
      m.mode = 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  p->tma_mode = m.mode;
  p->tm_wg = m.wg;
  p->tm_wu = m.wu;
  p->tm_wd = m.wd;
}

bool tma_plan(int w_dtype, int k, int d, int I, TmaPlan *plan) {
  if (w_dtype != DFV_BF16) return false;
  const int NT = k <= 8 ? 1 : 2;
  const size_t half = kSmemBudget / 2 + 1024;
  // gate/up: slice width ks = d / nslices with ks % 32 == 0 and ks <= 1024,
  // the widest such slice.  Two CTAs per SM when half the budget holds two
  // stages of it beside the two-token-tile x rows, else two CTAs per SM with
  // 512-column slices when those fit, else one CTA per SM.  ks sets how a
  // row's sum splits over the warps, so it depends on the shape only.
  const int C = d / 32;
  int nsl = (d + 1023) / 1024;
  while (nsl <= C && (C % nsl) != 0) ++nsl;
  if (nsl > C) return false;
  int ks = d / nsl, gper = 1;
  const size_t xg2 = (size_t)2 * 8 * pad_host(d * 2), redb2 = (size_t)kConsumerWarps * 2 * 32 * 16;
  auto two_fit = [&](int w) { return 1024 + (size_t)2 * 16 * pad_host(w * 2) + xg2 + redb2 + 32 <= half; };
  if (two_fit(ks)) {
    gper = 2;
  } else if (ks > 512 && d % 512 == 0 && two_fit(512)) {
    ks = 512;
    nsl = d / 512;
    gper = 2;
  }
  const size_t xg = (size_t)NT * 8 * pad_host(d * 2);
  const size_t redb = (size_t)kConsumerWarps * NT * 32 * 16;
  const size_t gbudget = gper == 2 ? half : kSmemBudget;
  int Sg = 4;
  size_t smg = 0;
  for (; Sg >= 2; --Sg) {
    smg = 1024 + (size_t)Sg * 16 * pad_host(ks * 2) + xg + redb + 16 * Sg;
    if (smg <= gbudget) break;
  }
  if (Sg < 2) return false;
  // down: rs rows of the full d_ff per stage.  rs sets how a row's sum splits
  // over the warps, so it is chosen for the largest block (two token tiles)
  // and is the same for every k: a block's rows then equal single-token calls
  // bit for bit.  The stage count then uses this block's own buffers.
  // two down CTAs per SM when a half budget holds two 16-row stages with the
  // two-token-tile buffers (the choice depends on the shape only, not on k);
  // else one CTA per SM with 32-row units when they fit
  const size_t hb2 = (size_t)2 * 8 * pad_host(I * 2);
  int rs = 16, per_sm = 2, dsl = 1;
  size_t budget = half;
  if (1024 + (size_t)2 * rs * pad_host(I * 2) + hb2 + redb2 + 32 > half) {
    if (I % 128 == 0 && 1024 + (size_t)2 * rs * pad_host(I) + hb2 + redb2 + 32 <= half) {
      dsl = 2;  // half of d_ff per stage keeps two CTAs per SM
    } else {
      per_sm = 1;
      budget = kSmemBudget;
      for (rs = 32; rs >= 16; rs /= 2)
        if ((size_t)2 * rs * pad_host(I * 2) + hb2 + redb2 + 32 <= kSmemBudget) break;
      if (rs < 16) return false;
    }
  }
  const size_t hb = (size_t)NT * 8 * pad_host(I * 2);
  int Sd = 4;
  size_t smd = 0;
  for (; Sd >= 2; --Sd) {
    smd = 1024 + (size_t)Sd * rs * pad_host(I * 2 / dsl) + hb + redb + 16 * Sd;
    if (smd <= budget) break;
  }
  if (Sd < 2) return false;
  plan->ks = ks;
  plan->nslices = nsl;
  plan->stages_g = Sg;
  plan->rs = rs;
  plan->stages_d = Sd;
  plan->down_per_sm = per_sm;
  plan->gate_per_sm = gper;
  plan->dsl = dsl;
  plan->smem_g = smg;
  plan->smem_d = smd;
  return true;
}

namespace {
template <typename F>
cudaError_t launch_tma(F kern, int grid, size_t smem, const FfnParams &p, cudaStream_t s, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
}  // namespace

cudaError_t launch_ffn_tma(const FfnParams &p0, int w_dtype, int phase, const TmaPlan &plan, int grid, cudaStream_t s,
                           bool pdl) {
  if (w_dtype != DFV_BF16) return cudaErrorInvalidValue;
  FfnParams p = p0;
  p.ks = plan.ks;
  p.nslices = plan.nslices;
  p.rs = plan.rs;
  if (phase == 0) {
    p.stages = plan.stages_g;
    return p.k <= 8 ? launch_tma(gateup_tma_kernel<1>, grid, plan.smem_g, p, s, pdl)
                    : launch_tma(gateup_tma_kernel<2>, grid, plan.smem_g, p, s, pdl);
  }
  if (phase == 2) {
    cudaLaunchConfig_t cfg = {};
    const int n = p.k * p.d;
    cfg.gridDim = dim3((n + 255) / 256 < 4 * grid ? (n + 255) / 256 : 4 * grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
  }
  p.stages = plan.stages_d;
  if (plan.dsl == 2)
    return p.k <= 8 ? launch_tma(down_tma_kernel<1, 2>, grid, plan.smem_d, p, s, pdl)
                    : launch_tma(down_tma_kernel<2, 2>, grid, plan.smem_d, p, s, pdl);
  return p.k <= 8 ? launch_tma(down_tma_kernel<1, 1>, grid, plan.smem_d, p, s, pdl)
                  : launch_tma(down_tma_kernel<2, 1>, grid, plan.smem_d, p, s, pdl);
}

}  // namespace dfv
