// layer_fused.cu -- one MoE layer of a verify block in a single persistent,
// cooperative launch (bf16 experts and router, bf16 activations).
//
// "Speculating on a Strix Halo", section "What the pieces cost": every token of
// the block routes to its own top-K experts and the block wakes their union;
// section "The verify's own cost": tokens are sorted by expert and each
// projection runs grouped.  Part 2, section "The verification cog": the cost is
// streaming the woken experts' weights, so every weight byte of a woken expert
// crosses HBM exactly once.
//
// One CTA per SM (grid = SM count, co-residency guaranteed by the cooperative
// launch); 16 consumer warps and one producer warp.  Before griddepcontrol.wait
// a CTA only starts its router rows towards L2.  Phases:
//   P0  router GEMV (optionally on RMSNorm(x) rounded to bf16): CTA b computes
//       the logits of experts b, b+G, ...; fixed-order reductions.  The idle
//       producer first copies the k rows of x into the staged-x rows, while
//       each warp's router row is in flight.
//       -- grid barrier 1 --
//   P1  every CTA derives the whole routing decision itself from the logits:
//       top-K per row (warp per row, redux max/min: largest logit, lowest id
//       among equals), routing weights, woken union, per-expert pair offsets
//       (block scan) and the (expert, token)-sorted pair list.  Each CTA
//       checks these tables before any phase indexes with them.  An
//       always-on shared expert (same section) joins them as the last woken
//       expert (id E), selected by every row with weight 1 (pairs k*K + t).
//   P2  gate/up: unit = (woken expert, 8 d_ff rows).  The producer streams
//       stages of 8 gate + 8 up rows x `ks` columns into an mbarrier ring (by
//       default one 3-D tensor copy per matrix in 128-byte segments with the
//       128-byte swizzle; 256-column boxes, or one bulk copy per row, on
//       request); the 16 consumer warps split the columns, run m16n8k16 MMAs
//       (gate rows = M 0-7, up rows = M 8-15, tokens = N; with the swizzle,
//       MMA row g is stored row (g >> 1) | ((g & 1) << 2), which keeps a
//       quarter-warp's fragment loads free of bank conflicts) and
//       reduce across warps in fixed order; h = silu(g) * u is written in
//       bf16.  The producer then runs ahead into P3's weights.
//       -- grid barrier 2 (consumers only) --
//   P3  down: unit = (woken expert, 16 d rows), expert-major and split into
//       contiguous ranges over the CTAs (so every SM works and a warp reuses
//       the h fragments of an expert across its tiles); each unit is one
//       contiguous copy; two groups of 8 warps take alternate units, reduce
//       within the group and write w[t,s] * y to ys[pair].  Each group owns
//       the ring stages of its parity, and every warp tracks each stage's
//       phase, so each parity wait is on a stage whose previous fill the
//       waiting warps consumed (with one shared odd-sized ring, a group could
//       pass a wait one phase early).
//       -- grid barrier 3 --
//   P4  every CTA sums ys over the K slots in slot order (then the shared
//       slot, + the residual) for its share of the outputs.  No atomics on
//       the output: the result of a token depends only on its own row, so a
//       block and k single-token calls agree bit for bit.
// Every wait is bounded (2 s) and reports through the workspace error word.
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "fused_common.cuh"

namespace dfv {

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// The kernel body.  STACK: `nl` layers of one shape in a row over the residual
// stream p.x (= p.out = p.residual), the weights of layer l in SL[l]; between
// layers a grid barrier (every row of x is combined) and the ring's mbarriers
// are armed afresh.  Without STACK, one layer with the weights in p.
// What the down phase reads besides the thread's own indexes.
struct DownArgs {
  const uint16_t *hbf;       // h rounded to bf16, [k*K][d_ff] by sorted pair position
  float *ys;                 // weighted expert outputs, by pair id
  unsigned *err;             // workspace error word
  const int *off, *gat;      // per woken expert: first sorted position; sorted pair ids
  const float *w;            // routing weight of each pair
  float *red;                // cross-warp reduction scratch [16][NT][32][4]
  volatile int *abort;
  uint32_t sbase, slot, full0, empty0, extra;  // ring, its barriers, the extra stage
  int SH, S, lo_d, hi_d, tiles_d, I, d;        // reserved and usable stages, this CTA's units
};

// P3: down = (woken expert, 16 d rows) units lo_d..hi_d-1 of this CTA,
// expert-major; two groups of 8 consumer warps take alternate units, reduce
// within the group and write w[t,s] * y to ys[pair].  Each group owns the
// ring stages of its parity.  Returns the updated stage phase bits; *dead is
// set when a wait gave up.
template <int NT>
__device__ __forceinline__ uint32_t down_phase(const DownArgs &A, uint32_t cbits, int *dead_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int I = A.I, d = A.d, S = A.S, SH = A.SH, tiles_d = A.tiles_d;
  const uint32_t full0 = A.full0, empty0 = A.empty0;
  const uint16_t *hbf = A.hbf;
  const int *s_off = A.off, *s_gat = A.gat;
  const float *s_w = A.w;
  bool dead = *dead_out != 0;
  auto slot_addr = [&](int st) -> uint32_t { return st < SH ? A.sbase + (uint32_t)st * A.slot : A.extra; };
  const int grp = warp >> 3, wg = warp & 7;
  const int C = I / 32;
  const int d0 = wg * C / 8, d1 = (wg + 1) * C / 8;
  const int rsd = I * 2;
  float *redg = A.red + grp * 8 * NT * 32 * 4;  // this group's [8][NT][32][4]
  int cur_d = -1, eoff = 0, em = 0;
  int gs = grp;  // this group's next stage (the group owns the stages of its parity)
  uint4 bh[3][NT];  // B fragments: h of the current expert's tokens (bf16), reused across its tiles
  // unit lo_d + j belongs to group j & 1
  for (int u = A.lo_d + grp; u < A.hi_d; u += 2) {
    const int s = gs;
    gs = (gs + 2 < S) ? gs + 2 : grp;
    const int wi = u / tiles_d, r0 = (u - wi * tiles_d) * 16;
    if (wi != cur_d) {
      // straight from L2, issued before the stage wait so the latencies overlap
      cur_d = wi;
      eoff = s_off[wi];
      em = s_off[wi + 1] - eoff;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          bh[j][nt] = make_uint4(0u, 0u, 0u, 0u);
          const int row = nt * 8 + g, ch = d0 + j;
          if (!dead && ch < d1 && row < em)
            bh[j][nt] = __ldcg(reinterpret_cast<const uint4 *>(hbf + (size_t)(eoff + row) * I + ch * 32 + c * 8));
        }
      }
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
    if (!dead && !mbar_wait_fast(full0 + 8 * s, (cbits >> s) & 1u, A.err, DFV_DEVERR_STAGE_WAIT, A.abort))
      dead = true;
    cbits ^= 1u << s;
    // A fragments chunk by chunk, each straight into its MMAs (holding all
    // three chunks' fragments would cost 16 more registers, and the stage
    // is released only a few MMAs later)
    if (!dead) {
      const uint32_t st = slot_addr(s);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        if (d0 + j < d1) {
          const uint32_t q16 = ((d0 + j) * 4 + c) * 16;
          const uint4 a0 = lds128(st + g * rsd + q16);
          const uint4 a1 = lds128(st + (g + 8) * rsd + q16);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt * 8 < em) {
              mma_bf16(acc[nt], a0.x, a1.x, a0.y, a1.y, bh[j][nt].x, bh[j][nt].y);
              mma_bf16(acc[nt], a0.z, a1.z, a0.w, a1.w, bh[j][nt].z, bh[j][nt].w);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_n(empty0 + 8 * s, 2);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4 *>(redg + ((wg * NT + nt) * 32 + lane) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    bar_sync_n(kBarGroup + grp, 256);
    const int gt = tid & 255;
    if (gt < NT * 128 && !dead) {
      const int q4 = gt & 3, ln = (gt >> 2) & 31, nt = gt >> 7;
      const int tok = nt * 8 + 2 * (ln & 3) + (q4 & 1);
      if (tok < em) {
        float y = 0.f;
        for (int w = 0; w < 8; ++w) y += redg[((w * NT + nt) * 32 + ln) * 4 + q4];
        const int pair = s_gat[eoff + tok];
        A.ys[(size_t)pair * d + r0 + (ln >> 2) + ((q4 & 2) ? 8 : 0)] = s_w[pair] * y;
      }
    }
    bar_sync_n(kBarGroup + grp, 256);
  }
  *dead_out = dead ? 1 : 0;
  return cbits;
}

template <int NT, bool STACK, bool SINGLE>
__device__ __forceinline__ void fused_body(const FusedParams &p, const StackLayer *SL, int nl) {
  pdl_trigger();
  prefetch_router_rows(STACK ? SL[0].wr : p.wr, p.E, p.d);
  pdl_wait();  // before this only the router-row prefetch touches global memory
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // 1024-aligned: the 128-byte swizzle of staging mode 3 repeats every 1024 bytes
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = p.k, d = p.d, I = p.I, K = p.K, ks = p.ks, nsl = p.nsl;
  const int G = gridDim.x;
  const int rsg = fpad(ks * 2);        // gate/up stage row stride (64 mod 128: conflict-free)
  const int rsx = d * 2;               // staged x row stride (16B chunks XOR-swizzled)
  // gate/up stage layout: padded rows (mode 0), [ks/256][8 rows][512 B] blocks
  // from tensor copies (modes 1, 2), or [ks/64][8 rows][128 B] segments with
  // the 128-byte swizzle (mode 3); up rows follow the gate rows
  const uint32_t row_b = p.tma_mode ? 512u : (uint32_t)rsg;
  const uint32_t blk_b = p.tma_mode ? 4096u : 512u;
  const uint32_t up_off = p.tma_mode ? 8u * ks * 2 : 8u * rsg;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t slot = p.slot;
  const int SH = p.ring;                                   // ring stages the launch reserved
  unsigned char *scratch = smem + SH * slot;               // x rows / logits / slot table
  float *red = reinterpret_cast<float *>(scratch + p.scratch);  // [16][NT][32][4]
  const uint32_t full0 = smem_u32(red + kFW * NT * 32 * 4);
  const uint32_t empty0 = full0 + 8 * kMaxRing;

  // routed pairs, then (with a shared expert) one shared pair per row
  __shared__ int s_idx[kMaxBlock * (kMaxTopK + 1)];
  __shared__ float s_w[kMaxBlock * (kMaxTopK + 1)];
  __shared__ int s_woken[kMaxExperts + 1];
  __shared__ int s_off[kMaxExperts + 2];
  __shared__ int s_eoff[kMaxExperts];
  __shared__ int s_gat[kMaxBlock * (kMaxTopK + 1)];
  __shared__ unsigned s_tmask[kMaxExperts];
  __shared__ float s_inv[kMaxBlock];
  __shared__ int s_tok[16];
  __shared__ int s_nw, s_ring, s_split;
  __shared__ volatile int s_abort, s_bad;
  __shared__ __align__(8) unsigned long long s_xbar;  // the copy of the k rows of x

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the k rows of x are copied into the staged-x rows (idle until gate/up),
  // which always hold at least k rows
  const uint32_t xbar = smem_u32(&s_xbar);
  auto init_bars = [&] {
    for (int s = 0; s <= SH; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kFW);
    }
    mbar_init(xbar, 1);
    mbar_init_fence();
  };
  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    init_bars();
  }
  __syncthreads();

  const bool consumer = warp < kFW;
#pragma unroll 1
  for (int l = 0; l < nl; ++l) {
  // (the layer's weights are read from the parameters where they are used)
  const unsigned gb = 4u * (unsigned)l;  // grid barriers completed before this layer
  if (STACK && l > 0) {
    // layer boundary: every CTA's combine has written its rows of x (the
    // writes are fenced for the async proxy, which copies x in next), and
    // every wait and copy on this CTA's mbarriers is over (the producer
    // drained its stages and the x copy), so they are armed afresh
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      if (!grid_sync(p, gb)) s_abort = 1;
      if (!s_abort) {
        for (int s = 0; s <= SH; ++s) {
          mbar_inval(full0 + 8 * s);
          mbar_inval(empty0 + 8 * s);
        }
        mbar_inval(xbar);
        init_bars();
      }
      s_bad = 0;
    }
    __syncthreads();
    if (s_abort) {
      // a CTA that gave up passes the later layers' grid barriers without
      // work (the others see the abort flag or time out)
      if (tid == 0)
        for (unsigned b = 1; b <= 3; ++b) grid_sync(p, gb + b);
      continue;
    }
  }
  if (!consumer && lane == 0) {
    if (STACK) asm volatile("fence.proxy.async.global;" ::: "memory");
    stage_x_rows(p, sbase + SH * slot, xbar);
    if (p.tma_mode) {
      prefetch_tensormap(STACK ? &SL[l].tm_wg : &p.tm_wg);
      prefetch_tensormap(STACK ? &SL[l].tm_wu : &p.tm_wu);
    }
  }
  // ------------------------------------------------------------------ P0, P1: routing
  if (consumer) {
    const RouteSmem rs = {s_idx, s_w, s_woken, s_off, s_eoff, s_gat, s_tmask, s_inv, &s_nw, &s_abort, &s_bad};
    RouteArgs ra = route_args(p, rs, reinterpret_cast<const uint16_t *>(scratch), xbar);
    if (STACK) {
      ra.wr = reinterpret_cast<const uint16_t *>(SL[l].wr);
      ra.u_nw = p.u_nw ? p.u_nw + l : nullptr;  // one count per layer
    }
    ra.gb = gb;
    route_p0(ra);
    route_p1<SINGLE>(ra, [&](int mmax) {
      // (warp 0, lane 0, right after the woken list is known; the producer
      // reads both words) with at most 8 tokens per gate/up entry the
      // staged-x rows 8..15 are unused: they become one more ring stage.  A
      // shared expert with more than 8 tokens then enters gate/up as two
      // entries (its rows 0-7 and 8-15), which reads its gate/up rows twice
      // but keeps that stage.  mmax: most tokens any routed expert took.
      const int nw0 = s_nw;
      const bool extra = NT == 2 && (uint32_t)p.scratch >= 8u * rsx + slot && SH < kMaxRing;
      const bool split = extra && p.ns && nw0 > 0 && k > 8 && mmax <= 8;
      if (p.ns && nw0 > 0 && !split) mmax = max(mmax, k);
      s_split = split ? 1 : 0;
      s_ring = (extra && mmax <= 8) ? SH + 1 : SH;
    });
  } else {
    bar_sync_n(kBarProducer, 64);  // released as soon as the woken list is known
  }

  const int nW = s_nw;  // 0 when the CTA aborted before its routing
  const int S = s_ring;
  // stage s lives in the reserved ring, or (s == SH) in staged-x rows 8..15
  auto slot_addr = [&](int st) -> uint32_t {
    return st < SH ? sbase + (uint32_t)st * slot : sbase + (uint32_t)SH * slot + 8u * rsx;
  };
  const int tiles_g = I / kGateTile;
  int lo_g, hi_g;
  {
    // gate/up entries: the woken experts, the shared one (last) possibly as
    // two halves of 8 tokens
    const int U = (nW + (nW > 0 ? s_split : 0)) * tiles_g;
    lo_g = (int)((unsigned)blockIdx.x * (unsigned)U / (unsigned)G);
    hi_g = (int)((unsigned)(blockIdx.x + 1) * (unsigned)U / (unsigned)G);
  }
  const int tiles_d = d / 16;
  int lo_d, hi_d;  // down units (woken expert, 16 d rows), expert-major, contiguous per CTA
  {
    const int U = nW * tiles_d;
    lo_d = (int)((unsigned)blockIdx.x * (unsigned)U / (unsigned)G);
    hi_d = (int)((unsigned)(blockIdx.x + 1) * (unsigned)U / (unsigned)G);
  }

  if (!consumer) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && !s_abort) {
      // the consumers read the x copy in the staged-x rows with generic loads,
      // and rows 8..15 may become a ring stage: order those reads before the
      // ring's async-proxy writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint64_t pol = l2_evict_first();  // expert weights are read once per launch
      const uint16_t *wg = reinterpret_cast<const uint16_t *>(STACK ? SL[l].wg : p.wg);
      const uint16_t *wu = reinterpret_cast<const uint16_t *>(STACK ? SL[l].wu : p.wu);
      const uint16_t *wd = reinterpret_cast<const uint16_t *>(STACK ? SL[l].wd : p.wd);
      const CUtensorMap *const tmg = STACK ? &SL[l].tm_wg : &p.tm_wg;
      const CUtensorMap *const tmu = STACK ? &SL[l].tm_wu : &p.tm_wu;
      // Stage phases are tracked per stage (bit s of pbits: parity of the next
      // fill's phase on stage s), because gate/up fills go round the whole
      // ring while down fills go round the stages of their consumer group.
      int ps = 0;
      uint32_t pbits = 0, used = 0;
      bool ok = true;
      for (int u = lo_g; u < hi_g && ok; ++u) {
        const int wi = u / tiles_g, i0 = (u % tiles_g) * kGateTile;
        const int e = s_woken[wi < s_nw ? wi : s_nw - 1];  // the second half: the shared expert again
        for (int sl = 0; sl < nsl; ++sl, ps = (ps + 1 == S) ? 0 : ps + 1) {
          const int s = ps;
          if (!mbar_wait_fast(empty0 + 8 * s, ((pbits >> s) & 1u) ^ 1u, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
            ok = false;
            break;
          }
          pbits ^= 1u << s;
          used |= 1u << s;
          const uint32_t fb = full0 + 8 * s, dst = slot_addr(s);
          mbar_expect_tx(fb, 16u * ks * 2);
          if (p.tma_mode == 3) {  // [ks/64][8 rows][128 B], swizzled: one box per matrix
            tma_3d_hint(dst, tmg, 0, e * I + i0, sl * (ks / 64), fb, pol);
            tma_3d_hint(dst + up_off, tmu, 0, e * I + i0, sl * (ks / 64), fb, pol);
          } else if (p.tma_mode == 2) {  // [ks/256][8 rows][256]: one box per matrix
            tma_3d_hint(dst, tmg, 0, e * I + i0, sl * (ks / 256), fb, pol);
            tma_3d_hint(dst + up_off, tmu, 0, e * I + i0, sl * (ks / 256), fb, pol);
          } else if (p.tma_mode == 1) {  // the same layout from 256-column boxes
            for (int b = 0; b < ks / 256; ++b) {
              tma_2d_hint(dst + b * 4096, tmg, sl * ks + b * 256, e * I + i0, fb, pol);
              tma_2d_hint(dst + up_off + b * 4096, tmu, sl * ks + b * 256, e * I + i0, fb, pol);
            }
          } else {  // one padded row per copy
            for (int r = 0; r < 8; ++r) {
              const size_t row = ((size_t)e * I + i0 + r) * d + (size_t)sl * ks;
              bulk_g2s_hint(dst + r * rsg, wg + row, ks * 2, fb, pol);
              bulk_g2s_hint(dst + (8 + r) * rsg, wu + row, ks * 2, fb, pol);
            }
          }
        }
      }
      // down unit lo_d + j belongs to consumer group j & 1, which owns the
      // stages of that parity: every wait on a stage then comes from warps
      // that consumed the stage's previous fill, so a parity wait can never be
      // taken for the phase before it
      int pg[2] = {0, 1};
      for (int u = lo_d, j = 0; u < hi_d && ok; ++u, ++j) {
        const int gq = j & 1, s = pg[gq];
        pg[gq] = (s + 2 < S) ? s + 2 : gq;
        if (!mbar_wait_fast(empty0 + 8 * s, ((pbits >> s) & 1u) ^ 1u, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
          ok = false;
          break;
        }
        pbits ^= 1u << s;
        used |= 1u << s;
        const int wi = u / tiles_d, tl = u - wi * tiles_d;
        const uint32_t fb = full0 + 8 * s;
        mbar_expect_tx(fb, 16u * I * 2);
        bulk_g2s_hint(slot_addr(s), wd + ((size_t)s_woken[wi] * d + (size_t)tl * 16) * I, 16u * I * 2, fb, pol);
      }
      if (STACK && l + 1 < nl) {
        // the next layer's router rows (this CTA's experts) and gate/up maps
        // start towards L2 and the descriptor cache while this layer drains
        const char *nwr = reinterpret_cast<const char *>(SL[l + 1].wr);
        for (int e = blockIdx.x; e < p.E; e += G) prefetch_l2(nwr + (size_t)e * d * 2, (uint32_t)d * 2);
        if (p.tma_mode) {
          prefetch_tensormap(&SL[l + 1].tm_wg);
          prefetch_tensormap(&SL[l + 1].tm_wu);
        }
      }
      // no copy may land after the CTA exits: wait for the last fill of every stage
      volatile int never = 0;
      for (int s = 0; s < S; ++s)
        if (((used >> s) & 1u) &&
            !mbar_wait(full0 + 8 * s, ((pbits >> s) & 1u) ^ 1u, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never))
          break;
    }
    if (lane == 0) {  // the x copy too (complete already unless a wait gave up)
      volatile int never = 0;
      mbar_wait(xbar, 0u, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never);
    }
  } else {
    // ---------------------------------------------------------------- P2: gate/up
    const int g = lane >> 2, c = lane & 3;
    const uint32_t pr = (uint32_t)((g >> 1) | ((g & 1) << 2));  // stored row of MMA row g (mode 3)
    const int cps = ks / 32;
    const int c0 = warp * cps / kFW, c1 = (warp + 1) * cps / kFW;
    const uint16_t *xg = reinterpret_cast<const uint16_t *>(p.x);
    const int cpr = d / 8;
    uint16_t *hbf = reinterpret_cast<uint16_t *>(p.ws.h);  // h rounded to bf16, [k*K][d_ff]
    const uint32_t xs = sbase + SH * slot;
    int cur = -1, m = 0, off = 0, cs = 0;  // cs: stage of the next gate/up fill
    uint32_t cbits = 0;                     // bit s: parity of the next phase of stage s
    bool dead = s_abort != 0;
    for (int u = lo_g; u < hi_g; ++u) {
      const int wi = u / tiles_g, i0 = (u % tiles_g) * kGateTile;
      if (wi != cur) {
        bar_sync_n(kBarAll, kFC);
        cur = wi;
        const int nr = s_nw - p.ns;  // routed experts; the shared one follows them
        if (wi < nr || !s_split) {
          off = s_off[wi];
          m = s_off[wi + 1] - off;
        } else {  // half wi - nr of the shared expert's k tokens
          off = s_off[nr] + 8 * (wi - nr);
          m = wi > nr ? p.k - 8 : 8;
        }
        if (tid < m) s_tok[tid] = pair_token(s_gat[off + tid], p.k, p.K);
        bar_sync_n(kBarAll, kFC);
        for (int idx = tid; idx < m * cpr; idx += kFC) {
          const int j = idx / cpr, q = idx % cpr, t = s_tok[j];
          // (a stack's later layers read rows other CTAs combined: from L2)
          const uint4 *src = reinterpret_cast<const uint4 *>(xg + (size_t)t * d + q * 8);
          uint4 v = STACK ? __ldcg(src) : *src;
          if (p.fuse_norm) {
            const float inv = s_inv[t];
            uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float a = rnd_bf16(bf16_lo(w4[h]) * inv), b = rnd_bf16(bf16_hi(w4[h]) * inv);
              w4[h] = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xffff0000u);
            }
            v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          *reinterpret_cast<uint4 *>(scratch + (size_t)j * rsx + ((q ^ ((j & 1) ? p.swz_x : 0)) * 16)) = v;
        }
        bar_sync_n(kBarAll, kFC);
      }
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
      for (int sl = 0; sl < nsl; ++sl, cs = (cs + 1 == S) ? 0 : cs + 1) {
        const int s = cs;
        if (!dead && !mbar_wait_fast(full0 + 8 * s, (cbits >> s) & 1u, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort))
          dead = true;
        cbits ^= 1u << s;
        // A fragments go to registers first and the slot is released at once,
        // so the producer refills it while the MMAs run
        uint4 ag[kMaxChunksP2], au[kMaxChunksP2];
        if (!dead) {
          const uint32_t st = slot_addr(s);
#pragma unroll
          for (int j = 0; j < kMaxChunksP2; ++j) {
            if (c0 + j < c1) {
              const int ch = c0 + j;  // 32-column chunk within the stage
              // mode 3: MMA row g reads stored row pr (rows 0,4,1,5,...), so the
              // two rows of a quarter-warp's loads sit in opposite halves of
              // the swizzle: no bank conflicts
              const uint32_t o = p.tma_mode == 3
                                     ? (ch >> 1) * 1024u + pr * 128u + ((((ch & 1) * 4 + c) ^ pr) << 4)
                                     : g * row_b + (ch >> 3) * blk_b + (ch & 7) * 64 + c * 16;
              ag[j] = lds128(st + o);
              au[j] = lds128(st + up_off + o);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (!dead) {
#pragma unroll
          for (int j = 0; j < kMaxChunksP2; ++j) {
            if (c0 + j < c1) {
              const int xq = sl * (ks / 8) + (c0 + j) * 4 + c;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt * 8 < m) {
                  const int row = nt * 8 + g;
                  uint4 b = make_uint4(0u, 0u, 0u, 0u);
                  if (row < m) b = lds128(xs + row * rsx + (xq ^ ((row & 1) ? p.swz_x : 0)) * 16);
                  mma_bf16(acc[nt], ag[j].x, au[j].x, ag[j].y, au[j].y, b.x, b.y);
                  mma_bf16(acc[nt], ag[j].z, au[j].z, ag[j].w, au[j].w, b.z, b.w);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4 *>(red + ((warp * NT + nt) * 32 + lane) * 4) =
            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      bar_sync_n(kBarAll, kFC);
      if (tid < NT * 64) {
        const int nt = tid >> 6, ln = (tid >> 1) & 31, q = tid & 1;
        const int tok = nt * 8 + 2 * (ln & 3) + q;
        if (tok < m) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kFW; ++w) {
            gs += red[((w * NT + nt) * 32 + ln) * 4 + q];
            us += red[((w * NT + nt) * 32 + ln) * 4 + q + 2];
          }
          const int gr = ln >> 2;  // MMA row; mode 3 stores it as row (gr >> 1) | ((gr & 1) << 2)
          const size_t o = (size_t)(off + tok) * I + i0 + (p.tma_mode == 3 ? ((gr >> 1) | ((gr & 1) << 2)) : gr);
          hbf[o] = __bfloat16_as_ushort(__float2bfloat16_rn(silu(gs) * us));
        }
      }
      bar_sync_n(kBarAll, kFC);
    }
    // ---- grid barrier 2: every h row is written
    if (tid == 0 && !grid_sync(p, gb + 2)) s_abort = 1;
    bar_sync_n(kBarAll, kFC);
    dead = dead || s_abort != 0;

    // ---------------------------------------------------------------- P3: down
    {
      const DownArgs da = {hbf, p.ws.ys, p.ws.err, s_off, s_gat, s_w, red, &s_abort,
                           sbase, slot, full0, empty0, sbase + (uint32_t)SH * slot + 8u * rsx,
                           SH, S, lo_d, hi_d, tiles_d, I, d};
      int dd = dead ? 1 : 0;
      cbits = down_phase<NT>(da, cbits, &dd);
      dead = dd != 0;
    }
    // ---- grid barrier 3: every ys row is written
    bar_sync_n(kBarAll, kFC);
    if (tid == 0 && !grid_sync(p, gb + 3)) s_abort = 1;
    bar_sync_n(kBarAll, kFC);
    dead = dead || s_abort != 0;

    // ---------------------------------------------------------------- P4: combine
    // out[t] = residual[t] + sum_s ys[t*K+s], slot order, + ys[k*K+t] (shared
    // expert), for this CTA's share of the outputs
    if (!dead) {
      const int n_out = k * d;
      const int o0 = (int)(((long long)blockIdx.x * n_out) / G), o1 = (int)(((long long)(blockIdx.x + 1) * n_out) / G);
      for (int o = o0 + tid; o < o1; o += kFC) {
        const int t = o / d, r = o - t * d;
        float sum = 0.f;
        for (int sl = 0; sl < K; ++sl) sum += __ldcg(p.ws.ys + (size_t)(t * K + sl) * d + r);
        if (p.ns) sum += __ldcg(p.ws.ys + (size_t)(k * K + t) * d + r);
        if (p.residual) sum = load_act(p.residual, (size_t)t * d + r, DFV_BF16) + sum;
        store_act(p.out, (size_t)t * d + r, DFV_BF16, sum);
      }
    }
  }
  }  // layers

  // exit ticket: the last CTA out resets the grid-barrier count for the next launch
  __syncthreads();
  if (tid == 0) {
    if (atomicAdd(p.ws.sync + 1, 1u) == (unsigned)(G - 1)) {
      atomicExch(p.ws.sync, 0u);
      atomicExch(p.ws.sync + 1, 0u);
    }
  }
}

// NT: token tiles of 8 (k <= 8: 1); SINGLE: instantiated for k = 1 only.
template <int NT, bool SINGLE>
__global__ void __launch_bounds__(kFT, 1) moe_fused_kernel(const __grid_constant__ FusedParams p) {
  fused_body<NT, false, SINGLE>(p, nullptr, 1);
}

// All layers of a residual stack in one persistent launch.
template <int NT, bool SINGLE>
__global__ void __launch_bounds__(kFT, 1) moe_stack_kernel(const __grid_constant__ StackParams sp) {
  fused_body<NT, true, SINGLE>(sp.p, sp.L, sp.n_layers);
}

// the instantiation for a block of k rows
template <bool STACK>
auto fused_kernel_for(int k) {
  if constexpr (STACK)
    return k == 1 ? moe_stack_kernel<1, true> : k <= 8 ? moe_stack_kernel<1, false> : moe_stack_kernel<2, false>;
  else
    return k == 1 ? moe_fused_kernel<1, true> : k <= 8 ? moe_fused_kernel<1, false> : moe_fused_kernel<2, false>;
}

// ----------------------------------------------------------------------------
// host side
bool fused_plan(int k, int d, int I, int E, FusedPlan *plan) {
  if (d % 32 || I % 32 || I > 768 || k < 1 || k > kMaxBlock) return false;  // P3 holds <= 3 k-chunks per warp
  const int NT = k <= 8 ? 1 : 2;
  const int C = d / 32;
  int nsl = (d + 1023) / 1024;
  while (nsl <= C && (C % nsl) != 0) ++nsl;
  if (nsl > C) return false;
  const int ks = d / nsl;
  if (ks / 32 > kFW * kMaxChunksP2) return false;
  auto pad = [](int b) { return (b % 128 == 0) ? b + 64 : b; };
  const size_t gslot = (size_t)16 * pad(ks * 2);
  const size_t dslot = (size_t)16 * I * 2;
  size_t slot = gslot > dslot ? gslot : dslot;
  slot = (slot + 1023) & ~(size_t)1023;  // stage bases 1024-aligned (the mode-3 swizzle)
  // staged x: NT * 8 rows.  k > 8: rows 8..15 double as one more ring stage
  // when no expert has more than 8 tokens, so they span at least one full slot
  size_t scratch = (size_t)NT * 8 * d * 2;
  if (NT == 2 && (size_t)8 * d * 2 + slot > scratch) scratch = (size_t)8 * d * 2 + slot;
  const size_t lgb = (size_t)k * E * 4, ysb = (size_t)k * 8 * 16 * 4;
  if (lgb > scratch) scratch = lgb;
  if (ysb > scratch) scratch = ysb;
  scratch = (scratch + 127) & ~(size_t)127;
  const size_t redb = (size_t)kFW * NT * 32 * 16;
  const size_t budget = 220 * 1024;
  int ring = 0;
  for (int r = kMaxRing - 1; r >= 4; --r) {
    if (1024 + r * slot + scratch + redb + 16 * kMaxRing <= budget) { ring = r; break; }
  }
  if (ring < 4) return false;
  plan->ks = ks;
  plan->nsl = nsl;
  plan->slot = (int)slot;
  plan->scratch = (int)scratch;
  plan->ring = ring;
  plan->smem = 1024 + ring * slot + scratch + redb + 16 * kMaxRing;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char *why, size_t why_len);

void fused_tensor_maps(FusedParams *p, const dfv_moe_layer *L, const FusedPlan &plan, int max_mode) {
  // the gate/up stage of 8 rows x ks columns as one swizzled 3-D box
  // ([ks/64][8][64], 128-byte swizzle: mode 3), one 3-D box ([ks/256][8][256]:
  // mode 2) or ks/256 2-D boxes of 8 x 256 (mode 1), the highest that max_mode
  // and the shape allow; cached per (weights, shape)
  struct Maps {
    int mode;
    CUtensorMap wg, wu;
  };
  static std::mutex mu;
  static std::map<std::tuple<const void *, const void *, int, int, int, int, int>, Maps> cache;
  p->tma_mode = 0;
  const int d = L->d, I = L->d_ff, E = L->n_experts + (L->n_shared ? 1 : 0), ks = plan.ks;  // the shared expert is the last
  if (d % 64 || ks % 64 || max_mode <= 0) return;
  const auto key = std::make_tuple(L->w_gate, L->w_up, d, I, E, ks, max_mode);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      p->tma_mode = it->second.mode;
      p->tm_wg = it->second.wg;
      p->tm_wu = it->second.wu;
      return;
    }
  }
  char why[128];
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, sizeof why);
  Maps m = {};
  if (fn) {
    const cuuint64_t rows = (cuuint64_t)E * I;
    auto enc3 = [&](CUtensorMap *map, const void *base) {
      const cuuint64_t dims[3] = {256, rows, (cuuint64_t)d / 256};
      const cuuint64_t strides[2] = {(cuuint64_t)d * 2, 512};
      const cuuint32_t box[3] = {256, 8, (cuuint32_t)ks / 256};
      const cuuint32_t es[3] = {1, 1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto enc2 = [&](CUtensorMap *map, const void *base) {
      const cuuint64_t dims[2] = {(cuuint64_t)d, rows};
      const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
      const cuuint32_t box[2] = {256, 8};
      const cuuint32_t es[2] = {1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto enc3s = [&](CUtensorMap *map, const void *base) {
      const cuuint64_t dims[3] = {64, rows, (cuuint64_t)d / 64};
      const cuuint64_t strides[2] = {(cuuint64_t)d * 2, 128};
      const cuuint32_t box[3] = {64, 8, (cuuint32_t)ks / 64};
      const cuuint32_t es[3] = {1, 1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (max_mode >= 3 && ks / 64 <= 256 && enc3s(&m.wg, L->w_gate) && enc3s(&m.wu, L->w_up))
      m.mode = 3;
    else if (d % 256 == 0 && ks % 256 == 0 && max_mode >= 2 && enc3(&m.wg, L->w_gate) && enc3(&m.wu, L->w_up))
      m.mode = 2;
    else if (d % 256 == 0 && ks % 256 == 0 && enc2(&m.wg, L->w_gate) && enc2(&m.wu, L->w_up))
      m.mode = 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  p->tma_mode = m.mode;
  p->tm_wg = m.wg;
  p->tm_wu = m.wu;
}

// Tensor maps and weight pointers of one layer of a stack launch; *mode is the
// staging mode the maps serve (every layer of a launch must share it).
bool stack_layer_maps(StackLayer *sl, const dfv_moe_layer *L, const FusedPlan &plan, int max_mode, int *mode) {
  FusedParams tmp = {};
  fused_tensor_maps(&tmp, L, plan, max_mode);
  sl->tm_wg = tmp.tm_wg;
  sl->tm_wu = tmp.tm_wu;
  sl->wr = L->w_router;
  sl->wg = L->w_gate;
  sl->wu = L->w_up;
  sl->wd = L->w_down;
  *mode = tmp.tma_mode;
  return true;
}

namespace {
// A cooperative launch (the grid barriers need every CTA resident), chained
// to the previous kernel programmatically when `pdl`: CTAs may start while it
// drains, and do nothing before griddepcontrol.wait.
template <class Kern, class Params>
cudaError_t launch_coop(Kern kern, const Params &p, size_t smem, int grid, cudaStream_t s, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFT);
  cfg.dynamicSmemBytes = smem;
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

// SM count when `kern` fits one CTA per SM with the plan's shared memory, else
// 0 with the reason in `why`.
template <class Kern>
int coop_max_grid(Kern kern, const FusedPlan &plan, char *why, size_t why_len) {
  int dev = 0, sms = 0, per = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    snprintf(why, why_len, "SM count query: %s", cudaGetErrorString(e));
    return 0;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(why, why_len, "shared memory %zu B: %s", plan.smem, cudaGetErrorString(e));
    return 0;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, kFT, plan.smem);
  if (e != cudaSuccess || per < 1) {
    cudaGetLastError();
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, kern);
    snprintf(why, why_len, "occupancy %d (%s): regs %d, static smem %zu, max threads %d, dyn smem %zu", per,
             cudaGetErrorString(e), fa.numRegs, fa.sharedSizeBytes, fa.maxThreadsPerBlock, plan.smem);
    return 0;
  }
  return sms;
}

void apply_plan(FusedParams &f, const FusedPlan &plan) {
  f.ks = plan.ks;
  f.nsl = plan.nsl;
  f.slot = plan.slot;
  f.scratch = plan.scratch;
  f.ring = plan.ring;
}
}  // namespace

cudaError_t launch_fused(const FusedParams &p0, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl) {
  FusedParams p = p0;
  apply_plan(p, plan);
  return launch_coop(fused_kernel_for<false>(p.k), p, plan.smem, grid, s, pdl);
}

cudaError_t launch_fused_stack(const StackParams &sp0, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl) {
  StackParams sp = sp0;
  apply_plan(sp.p, plan);
  return launch_coop(fused_kernel_for<true>(sp.p.k), sp, plan.smem, grid, s, pdl);
}

int fused_max_grid(const FusedPlan &plan, int k, char *why, size_t why_len) {
  return coop_max_grid(fused_kernel_for<false>(k), plan, why, why_len);
}

int fused_stack_max_grid(const FusedPlan &plan, int k, char *why, size_t why_len) {
  return coop_max_grid(fused_kernel_for<true>(k), plan, why, why_len);
}

}  // namespace dfv
