// layer_fused_mxfp4.cu -- one MoE layer of a verify block in a single
// persistent, cooperative launch, with mxfp4 expert weights (E2M1 codes and
// one E8M0 scale per 32 elements of a row; bf16 router, bf16 activations).
//
// "Speculating on a Strix Halo", sections "What the pieces cost" and "The
// verify's own cost": the block's tokens route to their own top-K experts, the
// block wakes their union, and tokens are grouped by expert.  The MI355X /
// vLLM write-up (allbreaknews.com/?p=4397), sections "Why Quantize the Target
// Model on Top?" and "Results: Quantizing the Target Model": the expert
// weights stay in fp4 all the way to the GEMM; here each woken expert's codes
// and scales cross HBM exactly once and are widened to fp16 in registers.
//
// One CTA per SM: 16 consumer warps in 4 groups of 4, and one producer warp
// that streams whole contiguous weight blocks through an 8-stage mbarrier ring
// (4 bulk copies per gate/up stage, 2 per down stage).  Group q consumes the
// stages q, q+4, q+8, ... of the ring sequence, so the groups run as four
// independent pipelines that synchronise only among their own 128 threads.
//   P0, P1  routing, shared with the bf16 single-launch kernel (fused_route).
//   P2  the k rows of x (after the optional RMSNorm, rounded to bf16) are
//       staged once in shared memory as fp16, each multiplied by a power of
//       two that puts its largest magnitude in [2^14, 2^15).  unit = (woken
//       expert, 8 d_ff rows); its stage holds the 8 gate and 8 up rows of codes
//       and their scales.  The group's 4 warps split d, widen their codes
//       (cvt e2m1x2 -> fp16x2, times the block scale), run m16n8k16 fp16 MMAs
//       (gate rows = M 0-7, up rows = M 8-15, the expert's tokens = N) and add
//       the 4 partial sums in fixed order; h = silu(g) * u goes to global
//       memory in fp32.
//       -- grid barrier 2 (consumers only; the producer runs ahead into P3) --
//   P3  unit = (woken expert, 64 d rows); its stage holds the 64 rows of down
//       codes and scales.  Each warp owns 16 rows over the whole d_ff; the B
//       operand is the expert's h rows, staged per expert in the group's
//       shared buffer as fp16 with their own power-of-two scales.
//       w[t,s] * y goes to ys[pair]; the last unit to finish a 64-row tile
//       (atomic ticket, nothing waits) sums ys over the K slots in slot order,
//       adds the residual and writes the output rows.  The sum order of every
//       output depends only on its own token, never on the block.
// Every wait is bounded (2 s) and reports through the workspace error word.
#include <cstdio>

#include "fused_common.cuh"
#include "mxfp4_common.cuh"

namespace dfv {
namespace {

constexpr int kMxRing = 8;               // ring stages (a power of two, a multiple of the groups)
constexpr int kMxGroups = 4;             // consumer groups
constexpr int kMxGW = kFW / kMxGroups;   // warps per group
constexpr int kMxBarGroup = 2;           // named barriers 2..5, one per group
constexpr int kMxMaxCh = 4;              // 128-code chunks per warp and row: d <= 2048, d_ff <= 512

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

template <int NT>
__global__ void __launch_bounds__(kFT, 1) moe_fused_mx_kernel(FusedParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char smem[];
  const int k = p.k, d = p.d, I = p.I, K = p.K;
  const int G = gridDim.x;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t slot = p.slot;
  unsigned char *scratch = smem + kMxRing * slot;                 // x rows (P2), h rows per group (P3)
  float *red = reinterpret_cast<float *>(scratch + p.scratch);    // [groups][4 warps][NT][32][4]
  const uint32_t full0 = smem_u32(red + kFW * NT * 32 * 4);
  const uint32_t empty0 = full0 + 8 * kMxRing;

  __shared__ int s_idx[kMaxBlock * kMaxTopK];
  __shared__ float s_w[kMaxBlock * kMaxTopK];
  __shared__ int s_woken[kMaxExperts];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_eoff[kMaxExperts];
  __shared__ int s_gat[kMaxBlock * kMaxTopK];
  __shared__ unsigned s_mask[kMaxBlock * (kMaxExperts / 32)];
  __shared__ float s_inv[kMaxBlock];
  __shared__ float s_xinv[kMaxBlock];             // 2^-shift of each staged x row
  __shared__ float s_hinv[kMxGroups][kMaxBlock];  // 2^-shift of each staged h row, per group
  __shared__ int s_wsum[kFW], s_csum[kFW];
  __shared__ int s_nw;
  __shared__ unsigned s_last[kMxGroups];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kMxRing; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kMxGW);
    }
    mbar_init_fence();
  }
  __syncthreads();

  const bool consumer = warp < kFW;
  if (consumer) {
    const RouteSmem rs = {s_idx, s_w, s_woken, s_off, s_eoff, s_gat, s_mask, s_inv, s_wsum, s_csum, &s_nw, &s_abort};
    fused_route(p, rs);
  }
  __syncthreads();  // routing tables visible to the producer

  const int nW = s_nw;
  const int tiles_g = I / 8, tiles_d = d / 64;
  int lo_g, hi_g, lo_d, hi_d;
  {
    const int U = nW * tiles_g, V = nW * tiles_d;
    lo_g = (int)(((long long)blockIdx.x * U) / G);
    hi_g = (int)(((long long)(blockIdx.x + 1) * U) / G);
    lo_d = (int)(((long long)blockIdx.x * V) / G);
    hi_d = (int)(((long long)(blockIdx.x + 1) * V) / G);
  }
  // stage layouts: gate/up = [8][d/2] gate codes | [8][d/2] up codes |
  // [8][d/32] gate scales | [8][d/32] up scales; down = [64][I/2] codes | [64][I/32] scales
  const uint32_t rowb_g = d / 2, srow_g = d / 32, rowb_d = I / 2, srow_d = I / 32;
  const uint32_t g_up = 8 * rowb_g, g_sc = 16 * rowb_g, g_scu = g_sc + 8 * srow_g, d_sc = 64 * rowb_d;
  const uint32_t bytes_g = 16 * rowb_g + 16 * srow_g, bytes_d = 64 * rowb_d + 64 * srow_d;

  if (!consumer) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && !s_abort) {
      const uint8_t *wg = reinterpret_cast<const uint8_t *>(p.wg);
      const uint8_t *wu = reinterpret_cast<const uint8_t *>(p.wu);
      const uint8_t *wd = reinterpret_cast<const uint8_t *>(p.wd);
      int it = 0, ps = 0, pph = 0;  // fills issued; slot and phase of the next fill
      bool ok = true;
      for (int u = lo_g; u < hi_g; ++u, ++it, ps = (ps + 1) & (kMxRing - 1), pph ^= (ps == 0)) {
        if (!mbar_wait_fast(empty0 + 8 * ps, pph ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
          ok = false;
          break;
        }
        const int wi = u / tiles_g;
        const size_t row = (size_t)s_woken[wi] * I + (size_t)(u - wi * tiles_g) * 8;
        const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * slot;
        mbar_expect_tx(fb, bytes_g);
        bulk_g2s(dst, wg + row * rowb_g, 8 * rowb_g, fb);
        bulk_g2s(dst + g_up, wu + row * rowb_g, 8 * rowb_g, fb);
        bulk_g2s(dst + g_sc, p.sg + row * srow_g, 8 * srow_g, fb);
        bulk_g2s(dst + g_scu, p.su + row * srow_g, 8 * srow_g, fb);
      }
      for (int u = lo_d; u < hi_d && ok; ++u, ++it, ps = (ps + 1) & (kMxRing - 1), pph ^= (ps == 0)) {
        if (!mbar_wait_fast(empty0 + 8 * ps, pph ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
          ok = false;
          break;
        }
        const int wi = u / tiles_d;
        const size_t row = (size_t)s_woken[wi] * d + (size_t)(u - wi * tiles_d) * 64;
        const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * slot;
        mbar_expect_tx(fb, bytes_d);
        bulk_g2s(dst, wd + row * rowb_d, 64 * rowb_d, fb);
        bulk_g2s(dst + d_sc, p.sd + row * srow_d, 64 * srow_d, fb);
      }
      // no copy may land after the CTA exits
      volatile int never = 0;
      for (int j = it - kMxRing < 0 ? 0 : it - kMxRing; j < it; ++j)
        if (!mbar_wait(full0 + 8 * (j % kMxRing), (j / kMxRing) & 1, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never)) break;
    }
  } else {
    const int grp = warp / kMxGW, wq = warp % kMxGW, gt = tid % (kMxGW * 32);
    const int g = lane >> 2, c = lane & 3;
    const int bar_grp = kMxBarGroup + grp;
    float *redg = red + grp * (kMxGW * NT * 32 * 4);
    float *hf = p.ws.h;  // [k*K][I] fp32, by sorted pair position
    uint32_t bad = 0;
    bool dead = s_abort != 0;

    // ---- stage the k rows of x as fp16 (warp t: row t)
    const uint32_t xs = smem_u32(scratch);
    const int cpr = d / 8;
    if (warp < k) {
      const int t = warp;
      const uint16_t *src = reinterpret_cast<const uint16_t *>(p.x) + (size_t)t * d;
      const float inv = p.fuse_norm ? s_inv[t] : 1.f;
      float amax = 0.f;
      for (int q = lane; q < cpr; q += 32) {
        float f[8];
        load8_bf16(src, (size_t)q * 8, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(p.fuse_norm ? rnd_bf16(f[i] * inv) : f[i]));
      }
      const int sh = row_shift(warp_max(amax));
      const float sc = exp2i(sh);
      for (int q = lane; q < cpr; q += 32) {
        float f[8];
        load8_bf16(src, (size_t)q * 8, f);
        if (p.fuse_norm) {
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = rnd_bf16(f[i] * inv);
        }
        *reinterpret_cast<uint4 *>(scratch + (size_t)t * d * 2 + swz(q, t) * 16) =
            make_uint4(pack_h2(f[0] * sc, f[1] * sc), pack_h2(f[2] * sc, f[3] * sc), pack_h2(f[4] * sc, f[5] * sc),
                       pack_h2(f[6] * sc, f[7] * sc));
      }
      if (lane == 0) s_xinv[t] = exp2i(-sh);
    }
    bar_sync_n(kBarAll, kFC);

    // ---------------------------------------------------------------- P2: gate/up
    const int C = (d + 127) / 128;
    const int c0 = wq * C / kMxGW, c1 = (wq + 1) * C / kMxGW;
    int cs = grp, cph = 0;  // ring slot and phase of this group's next stage
    for (int u = lo_g + grp; u < hi_g; u += kMxGroups) {
      const int wi = u / tiles_g, i0 = (u - wi * tiles_g) * 8;
      const int off = s_off[wi], m = s_off[wi + 1] - off;
      if (!dead && !mbar_wait_fast(full0 + 8 * cs, cph, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) dead = true;
      // codes and scales to registers, then the stage is released at once
      uint4 ag[kMxMaxCh], au[kMxMaxCh];
      uint32_t eg[kMxMaxCh], eu[kMxMaxCh];
      const uint32_t st = sbase + cs * slot;
#pragma unroll
      for (int j = 0; j < kMxMaxCh; ++j) {
        const int ch = c0 + j;
        ag[j] = au[j] = make_uint4(0u, 0u, 0u, 0u);
        eg[j] = eu[j] = 127u;
        if (!dead && ch < c1 && ch * 128 + c * 32 < d) {
          const uint32_t o = g * rowb_g + ch * 64 + c * 16;
          ag[j] = lds128(st + o);
          au[j] = lds128(st + g_up + o);
          eg[j] = lds_u8(st + g_sc + g * srow_g + ch * 4 + c);
          eu[j] = lds_u8(st + g_scu + g * srow_g + ch * 4 + c);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * cs);
      cs += kMxGroups;
      if (cs >= kMxRing) {
        cs -= kMxRing;
        cph ^= 1;
      }
      int trow[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        trow[nt] = n < m ? s_gat[off + n] / K : -1;
      }
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
      if (!dead) {
#pragma unroll
        for (int j = 0; j < kMxMaxCh; ++j) {
          const int ch = c0 + j;
          if (ch < c1) {
            const bool live = ch * 128 + c * 32 < d;
            const uint32_t sgv = e8m0_half2(eg[j], bad), suv = e8m0_half2(eu[j], bad);
            const uint32_t wg4[4] = {ag[j].x, ag[j].y, ag[j].z, ag[j].w};
            const uint32_t wu4[4] = {au[j].x, au[j].y, au[j].z, au[j].w};
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
              uint32_t rg4[4], ru4[4];
              mx_decode_word(wg4[tt], sgv, rg4);
              mx_decode_word(wu4[tt], suv, ru4);
              const int q = ch * 16 + c * 4 + tt;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt * 8 < m) {
                  uint4 b = make_uint4(0u, 0u, 0u, 0u);
                  if (trow[nt] >= 0 && live) b = lds128(xs + trow[nt] * (d * 2) + swz(q, trow[nt]) * 16);
                  mma_f16x(acc[nt], rg4[0], ru4[0], rg4[1], ru4[1], b.x, b.y);
                  mma_f16x(acc[nt], rg4[2], ru4[2], rg4[3], ru4[3], b.z, b.w);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4 *>(redg + ((wq * NT + nt) * 32 + lane) * 4) =
            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      bar_sync_n(bar_grp, kMxGW * 32);
      if (gt < NT * 64 && !dead) {
        const int nt = gt >> 6, ln = (gt >> 1) & 31, q = gt & 1;
        const int tok = nt * 8 + 2 * (ln & 3) + q;
        if (tok < m) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kMxGW; ++w) {
            gs += redg[((w * NT + nt) * 32 + ln) * 4 + q];
            us += redg[((w * NT + nt) * 32 + ln) * 4 + q + 2];
          }
          const float inv = s_xinv[s_gat[off + tok] / K];
          hf[(size_t)(off + tok) * I + i0 + (ln >> 2)] = silu(gs * inv) * (us * inv);
        }
      }
      bar_sync_n(bar_grp, kMxGW * 32);
    }
    // ---- grid barrier 2: every h row is written (and the staged x is dead)
    bar_sync_n(kBarAll, kFC);
    if (tid == 0 && !grid_sync(p, 2)) s_abort = 1;
    bar_sync_n(kBarAll, kFC);
    dead = dead || s_abort != 0;

    // ---------------------------------------------------------------- P3: down + combine
    const int CI = (I + 127) / 128;
    const int hcpr = I / 8;
    unsigned char *hrows = scratch + (size_t)grp * (NT * 8) * I * 2;  // this group's staged h rows
    const uint32_t hb = smem_u32(hrows);
    const int nP2 = hi_g - lo_g;
    int cur = -1, m = 0, off = 0;
    for (int u = lo_d + (((grp - nP2) % kMxGroups) + kMxGroups) % kMxGroups; u < hi_d; u += kMxGroups) {
      const int wi = u / tiles_d, dt = u - wi * tiles_d;
      if (wi != cur) {
        bar_sync_n(bar_grp, kMxGW * 32);  // the previous expert's h rows are no longer read
        cur = wi;
        off = s_off[wi];
        m = s_off[wi + 1] - off;
        for (int n = wq; n < m; n += kMxGW) {
          const float *src = hf + (size_t)(off + n) * I;
          float amax = 0.f;
          for (int q = lane; q < hcpr; q += 32) {
            const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8));
            const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8 + 4));
            amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                                     fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w)))));
          }
          const int sh = row_shift(warp_max(amax));
          const float sc = exp2i(sh);
          for (int q = lane; q < hcpr; q += 32) {
            const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8));
            const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8 + 4));
            *reinterpret_cast<uint4 *>(hrows + (size_t)n * I * 2 + swz(q, n) * 16) =
                make_uint4(pack_h2(v0.x * sc, v0.y * sc), pack_h2(v0.z * sc, v0.w * sc),
                           pack_h2(v1.x * sc, v1.y * sc), pack_h2(v1.z * sc, v1.w * sc));
          }
          if (lane == 0) s_hinv[grp][n] = exp2i(-sh);
        }
        bar_sync_n(bar_grp, kMxGW * 32);
      }
      if (!dead && !mbar_wait_fast(full0 + 8 * cs, cph, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) dead = true;
      uint4 a0[kMxMaxCh], a1[kMxMaxCh];
      uint32_t e0[kMxMaxCh], e1[kMxMaxCh];
      const uint32_t st = sbase + cs * slot;
      const int rr = wq * 16 + g;
#pragma unroll
      for (int j = 0; j < kMxMaxCh; ++j) {
        a0[j] = a1[j] = make_uint4(0u, 0u, 0u, 0u);
        e0[j] = e1[j] = 127u;
        if (!dead && j < CI && j * 128 + c * 32 < I) {
          const uint32_t o = rr * rowb_d + j * 64 + c * 16;
          a0[j] = lds128(st + o);
          a1[j] = lds128(st + o + 8 * rowb_d);
          e0[j] = lds_u8(st + d_sc + rr * srow_d + j * 4 + c);
          e1[j] = lds_u8(st + d_sc + (rr + 8) * srow_d + j * 4 + c);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * cs);
      cs += kMxGroups;
      if (cs >= kMxRing) {
        cs -= kMxRing;
        cph ^= 1;
      }
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
      if (!dead) {
#pragma unroll
        for (int j = 0; j < kMxMaxCh; ++j) {
          if (j < CI) {
            const bool live = j * 128 + c * 32 < I;
            const uint32_t s0 = e8m0_half2(e0[j], bad), s1 = e8m0_half2(e1[j], bad);
            const uint32_t w0[4] = {a0[j].x, a0[j].y, a0[j].z, a0[j].w};
            const uint32_t w1[4] = {a1[j].x, a1[j].y, a1[j].z, a1[j].w};
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
              uint32_t r0v[4], r1v[4];
              mx_decode_word(w0[tt], s0, r0v);
              mx_decode_word(w1[tt], s1, r1v);
              const int q = j * 16 + c * 4 + tt;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt * 8 < m) {
                  const int n = nt * 8 + g;
                  uint4 b = make_uint4(0u, 0u, 0u, 0u);
                  if (n < m && live) b = lds128(hb + n * (I * 2) + swz(q, n) * 16);
                  mma_f16x(acc[nt], r0v[0], r1v[0], r0v[1], r1v[1], b.x, b.y);
                  mma_f16x(acc[nt], r0v[2], r1v[2], r0v[3], r1v[3], b.z, b.w);
                }
              }
            }
          }
        }
      }
      const int r0 = dt * 64 + wq * 16;
      if (!dead) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int tok = nt * 8 + 2 * c + q;
            if (tok < m) {
              const int pair = s_gat[off + tok];
              const float w = s_w[pair] * s_hinv[grp][tok];
              p.ws.ys[(size_t)pair * d + r0 + g] = w * acc[nt][q];
              p.ws.ys[(size_t)pair * d + r0 + g + 8] = w * acc[nt][q + 2];
            }
          }
      }
      // tile ticket: the last of the nW experts to finish tile dt combines it
      __threadfence();
      bar_sync_n(bar_grp, kMxGW * 32);
      if (gt == 0) s_last[grp] = (atomicAdd(p.ws.down_cnt + dt, 1u) == (unsigned)(nW - 1)) ? 1u : 0u;
      bar_sync_n(bar_grp, kMxGW * 32);
      if (s_last[grp]) {
        __threadfence();
        if (!dead) {
          for (int idx = gt; idx < k * 64; idx += kMxGW * 32) {
            const int t = idx >> 6, r = dt * 64 + (idx & 63);
            float sum = 0.f;
            for (int sl = 0; sl < K; ++sl) sum += __ldcg(p.ws.ys + (size_t)(t * K + sl) * d + r);
            if (p.residual) sum = load_act(p.residual, (size_t)t * d + r, DFV_BF16) + sum;
            store_act(p.out, (size_t)t * d + r, DFV_BF16, sum);
          }
        }
        if (gt == 0) p.ws.down_cnt[dt] = 0u;
      }
    }
    if (bad) atomicOr(p.ws.err, DFV_DEVERR_SCALE_RANGE);
  }

  // exit ticket: the last CTA out resets the grid-barrier count for the next launch
  __syncthreads();
  if (tid == 0) {
    if (atomicAdd(p.ws.sync + 1, 1u) == (unsigned)(G - 1)) {
      atomicExch(p.ws.sync, 0u);
      atomicExch(p.ws.sync + 1, 0u);
    }
  }
}

template <int NT>
size_t mx_smem(int d, int I, size_t *slot_out, size_t *scratch_out) {
  size_t gslot = (size_t)8 * d + d / 2, dslot = (size_t)34 * I;
  size_t slot = gslot > dslot ? gslot : dslot;
  slot = (slot + 127) & ~(size_t)127;
  size_t xsb = (size_t)NT * 8 * d * 2, hsb = (size_t)kMxGroups * NT * 8 * I * 2;
  size_t scratch = xsb > hsb ? xsb : hsb;
  scratch = (scratch + 127) & ~(size_t)127;
  *slot_out = slot;
  *scratch_out = scratch;
  return kMxRing * slot + scratch + (size_t)kFW * NT * 32 * 16 + 16 * kMxRing;
}

}  // namespace

// ----------------------------------------------------------------------------
// host side
bool fused_mx_plan(int k, int d, int I, int E, FusedPlan *plan) {
  if (k < 1 || k > kMaxBlock || E < 1 || E > kMaxExperts) return false;
  if (d % 64 || I % 64 || d > 128 * kMxMaxCh * kMxGW || I > 128 * kMxMaxCh) return false;
  size_t slot = 0, scratch = 0;
  const size_t smem = k <= 8 ? mx_smem<1>(d, I, &slot, &scratch) : mx_smem<2>(d, I, &slot, &scratch);
  if (smem > 220 * 1024) return false;
  plan->ks = 0;
  plan->nsl = 0;
  plan->slot = (int)slot;
  plan->scratch = (int)scratch;
  plan->ring = kMxRing;
  plan->smem = smem;
  return true;
}

cudaError_t launch_fused_mx(const FusedParams &p0, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl) {
  FusedParams p = p0;
  p.slot = plan.slot;
  p.scratch = plan.scratch;
  p.ring = plan.ring;
  auto kern = p.k <= 8 ? moe_fused_mx_kernel<1> : moe_fused_mx_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFT);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

int fused_mx_max_grid(const FusedPlan &plan, int k, char *why, size_t why_len) {
  int dev = 0, sms = 0, per = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    snprintf(why, why_len, "SM count query: %s", cudaGetErrorString(e));
    return 0;
  }
  auto kern = k <= 8 ? moe_fused_mx_kernel<1> : moe_fused_mx_kernel<2>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(why, why_len, "mxfp4: shared memory %zu B: %s", plan.smem, cudaGetErrorString(e));
    return 0;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, kFT, plan.smem);
  if (e != cudaSuccess || per < 1) {
    cudaGetLastError();
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, kern);
    snprintf(why, why_len, "mxfp4: occupancy %d (%s): regs %d, static smem %zu, max threads %d, dyn smem %zu", per,
             cudaGetErrorString(e), fa.numRegs, fa.sharedSizeBytes, fa.maxThreadsPerBlock, plan.smem);
    return 0;
  }
  return sms;
}

}  // namespace dfv
