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
// that streams the weights through an 8-stage mbarrier ring (4 tensor copies
// per gate/up stage, 2 bulk copies per down stage).  The producer feeds the
// groups round-robin, so group q consumes stages q, q+4, q+8, ... (a group with
// no unit left in a round gets an empty stage); no warp ever waits for another
// warp's partial sums.
//   P0, P1  routing, shared with the bf16 single-launch kernel (route_p0,
//       route_p1, on the k rows of x the producer copies into the staged-x
//       rows at the start; the producer starts streaming as soon as the woken
//       list is known);
//       an always-on shared expert ("What the pieces cost") joins the tables
//       as the last woken expert, which every row selects with weight 1.
//   P2  the k rows of x (after the optional RMSNorm, rounded to bf16) become
//       fp16 in place in shared memory, each multiplied by a power of two that
//       puts its largest magnitude in [2^14, 2^15), while the first stages
//       are in flight.  unit = (woken
//       expert, 32 d_ff rows), streamed as d/512 stages of 32 gate rows and
//       32 up rows x 512 codes with their scales (2-D tensor copies).  Warp w
//       of the group owns rows 8w..8w+7 over the whole of d: it widens its
//       codes (cvt e2m1x2 -> fp16x2, times the block scale), runs m16n8k16 fp16
//       MMAs (gate rows = M 0-7, up rows = M 8-15, the expert's tokens = N) and
//       keeps the sums in its registers across the stages; h = silu(g) * u goes
//       to global memory in fp32.  When all its gate/up units are done, the CTA
//       sets its own flag in the workspace with one release.  No grid barrier
//       follows: the producer runs straight on into P3's weights.
//   P3  unit = (woken expert, 64 d rows); its stage holds the 64 rows of down
//       codes and scales.  Before it first reads an expert's h, a group waits
//       (acquire, bounded) for the flags of the CTAs that own that expert's
//       gate/up units, polled by a whole warp at once.  Each warp owns 16 rows
//       over the whole d_ff; the B operand is the expert's h rows, staged per
//       expert in the group's shared buffer as fp16 with their own
//       power-of-two scales.  w[t,s] * y goes to ys[pair].
//       -- grid barrier 2 --
//   P4  every CTA sums ys over the K slots in slot order (then the shared
//       slot) for its share of the output rows, adds the residual and writes
//       them.  The sum order of
//       every output depends only on its own token, never on the block.
// Every wait is bounded (2 s) and reports through the workspace error word.
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "fused_common.cuh"
#include "mxfp4_common.cuh"

namespace dfv {
namespace {

constexpr int kMxGroups = 4;             // consumer groups
constexpr int kMxGW = kFW / kMxGroups;   // warps per group
constexpr int kMxRing = 8;               // ring stages (two per group)
constexpr int kMxBarGroup = 2;           // named barriers 2..5, one per group
constexpr int kMxCh = 4;                 // 128-code chunks per warp, row and stage
constexpr int kMxRows = 32;              // d_ff rows per gate/up unit (8 per warp)
constexpr int kMxCols = 512;             // codes per row and gate/up stage
constexpr int kMxMaxD = 2048;            // staged x: at most 8 16-byte pieces per lane

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// 2-D tensor copy global -> shared (box given by the tensor map), completion
// counted in bytes on `bar`.  x is the innermost (byte) coordinate.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Bounded wait, by one whole warp, until CTAs b0..b1 have published the end of
// their gate/up work (every h row they own is written): lane l polls CTAs
// b0 + l, b0 + l + 32, ... so the flags are read in parallel.
static __device__ __noinline__ bool ctas_done(const unsigned *flags, int b0, int b1, unsigned *err,
                                              volatile int *abort) {
  const int lane = threadIdx.x & 31;
  const unsigned long long t0 = global_ns();
  bool ok = true;
  for (int b = b0 + lane; b <= b1 && ok; b += 32) {
    // one load per poll; the abort flag and the clock every 16th poll
    for (unsigned it = 1; ld_acquire(flags + b) == 0u; ++it) {
      if ((it & 15u) == 0 && (*abort || global_ns() - t0 > kWaitNs)) {
        if (!*abort) atomicOr(err, DFV_DEVERR_GRID_WAIT);
        *abort = 1;
        ok = false;
        break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

template <int NT>
__global__ void __launch_bounds__(kFT, 1) moe_fused_mx_kernel(const __grid_constant__ FusedParams p) {
  pdl_trigger();
  prefetch_router_rows(p);
  pdl_wait();  // before this only the router-row prefetch touches global memory
  extern __shared__ __align__(128) unsigned char smem[];
  const int k = p.k, d = p.d, I = p.I, K = p.K;
  const int G = gridDim.x;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t slot = p.slot;
  unsigned char *scratch = smem + kMxRing * slot;  // x rows (P2), h rows per group (P3)
  const uint32_t full0 = sbase + kMxRing * slot + p.scratch;
  const uint32_t empty0 = full0 + 8 * kMxRing;
  float *acc1s = reinterpret_cast<float *>(smem + kMxRing * slot + p.scratch + 16 * kMxRing);  // [16 warps][32][4]
  // plain C++ loads from shared memory (ordered by the compiler against the
  // barrier waits, free to be scheduled early otherwise)
  auto ld16 = [&](uint32_t a) { return *reinterpret_cast<const uint4 *>(smem + (a - sbase)); };
  auto ld1 = [&](uint32_t a) { return (uint32_t)smem[a - sbase]; };

  // routed pairs, then (with a shared expert) one shared pair per row
  __shared__ int s_idx[kMaxBlock * (kMaxTopK + 1)];
  __shared__ float s_w[kMaxBlock * (kMaxTopK + 1)];
  __shared__ int s_woken[kMaxExperts + 1];
  __shared__ int s_off[kMaxExperts + 2];
  __shared__ int s_eoff[kMaxExperts];
  __shared__ int s_gat[kMaxBlock * (kMaxTopK + 1)];
  __shared__ unsigned s_tmask[kMaxExperts];
  __shared__ float s_inv[kMaxBlock];
  __shared__ float s_xinv[kMaxBlock];             // 2^-shift of each staged x row
  __shared__ float s_hinv[kMxGroups][kMaxBlock];  // 2^-shift of each staged h row, per group
  __shared__ int s_nw;
  __shared__ unsigned s_last_cta;
  __shared__ volatile int s_abort, s_bad;
  __shared__ __align__(8) unsigned long long s_xbar;  // the copy of the k rows of x

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t xbar = smem_u32(&s_xbar);
  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    for (int s = 0; s < kMxRing; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kMxGW);
    }
    mbar_init(xbar, 1);
    mbar_init_fence();
  }
  __syncthreads();

  const bool consumer = warp < kFW;
  if (!consumer && lane == 0) {
    // the producer is idle until the routing is known: it copies the k rows
    // of x into the staged-x rows and warms the tensor maps
    stage_x_rows(p, smem_u32(scratch), xbar);
    prefetch_tensormap(&p.tm_wg);
    prefetch_tensormap(&p.tm_wu);
    prefetch_tensormap(&p.tm_sg);
    prefetch_tensormap(&p.tm_su);
  }
  if (consumer) {
    const RouteSmem rs = {s_idx, s_w, s_woken, s_off, s_eoff, s_gat, s_tmask, s_inv, &s_nw, &s_abort, &s_bad};
    const RouteArgs ra = route_args(p, rs, reinterpret_cast<const uint16_t *>(scratch), xbar);
    route_p0(ra);
    route_p1(ra, [] {});
  } else {
    bar_sync_n(kBarProducer, 64);  // released as soon as the woken list is known
  }

  const int nW = s_nw;  // 0 when the CTA aborted before its routing
  const int tiles_g = I / kMxRows, tiles_d = d / 64, nq = d / kMxCols;
  int lo_g, hi_g, lo_d, hi_d;
  {
    const int U = nW * tiles_g, V = nW * tiles_d;
    lo_g = (int)((unsigned)blockIdx.x * (unsigned)U / (unsigned)G);
    hi_g = (int)((unsigned)(blockIdx.x + 1) * (unsigned)U / (unsigned)G);
    lo_d = (int)((unsigned)blockIdx.x * (unsigned)V / (unsigned)G);
    hi_d = (int)((unsigned)(blockIdx.x + 1) * (unsigned)V / (unsigned)G);
  }
  const int R2 = (hi_g - lo_g + kMxGroups - 1) / kMxGroups, R3 = (hi_d - lo_d + kMxGroups - 1) / kMxGroups;
  // stage layouts: gate/up = [32][256] gate codes | [32][256] up codes |
  // [32][16] gate scales | [32][16] up scales; down = [64][I/2] codes | [64][I/32] scales
  constexpr uint32_t g_up = kMxRows * kMxCols / 2, g_sc = 2 * g_up, g_scu = g_sc + kMxRows * kMxCols / 32;
  constexpr uint32_t bytes_g = 2 * g_up + 2 * kMxRows * kMxCols / 32;
  const uint32_t rowb_d = I / 2, srow_d = I / 32, d_sc = 64 * rowb_d;
  const uint32_t bytes_d = 64 * rowb_d + 64 * srow_d;

  if (!consumer) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && !s_abort) {
      const uint64_t pol = l2_evict_first();  // expert weights are read once per launch
      const uint8_t *wd = reinterpret_cast<const uint8_t *>(p.wd);
      int it = 0, ps = 0, pph = 0;  // stages issued; slot and phase of the next one
      bool ok = true;
      auto take = [&]() -> bool {
        if (!mbar_wait_fast(empty0 + 8 * ps, pph ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) return false;
        return true;
      };
      auto advance = [&]() {
        ++it;
        if (++ps == kMxRing) {
          ps = 0;
          pph ^= 1;
        }
      };
      // gate/up: rounds of one unit per group, d/512 stages per unit
      for (int r = 0; r < R2 && ok; ++r) {
        for (int q = 0; q < nq && ok; ++q) {
          for (int gq = 0; gq < kMxGroups; ++gq) {
            if (!take()) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * slot;
            const int u = lo_g + r * kMxGroups + gq;
            if (u < hi_g) {
              const int wi = u / tiles_g;
              const int row = s_woken[wi] * I + (u - wi * tiles_g) * kMxRows;
              mbar_expect_tx(fb, bytes_g);
              tma_2d_hint(dst, &p.tm_wg, q * (kMxCols / 2), row, fb, pol);
              tma_2d_hint(dst + g_up, &p.tm_wu, q * (kMxCols / 2), row, fb, pol);
              tma_2d_hint(dst + g_sc, &p.tm_sg, q * (kMxCols / 32), row, fb, pol);
              tma_2d_hint(dst + g_scu, &p.tm_su, q * (kMxCols / 32), row, fb, pol);
            } else {
              mbar_arrive(fb);  // empty stage: this group has no unit in this round
            }
            advance();
          }
        }
      }
      // down: rounds of one unit per group
      for (int r = 0; r < R3 && ok; ++r) {
        for (int gq = 0; gq < kMxGroups; ++gq) {
          if (!take()) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * slot;
          const int u = lo_d + r * kMxGroups + gq;
          if (u < hi_d) {
            const int wi = u / tiles_d;
            const size_t row = (size_t)s_woken[wi] * d + (size_t)(u - wi * tiles_d) * 64;
            mbar_expect_tx(fb, bytes_d);
            bulk_g2s_hint(dst, wd + row * rowb_d, 64 * rowb_d, fb, pol);
            bulk_g2s_hint(dst + d_sc, p.sd + row * srow_d, 64 * srow_d, fb, pol);
          } else {
            mbar_arrive(fb);
          }
          advance();
        }
      }
      // no copy may land after the CTA exits
      volatile int never = 0;
      for (int j = it - kMxRing < 0 ? 0 : it - kMxRing; j < it; ++j)
        if (!mbar_wait(full0 + 8 * (j % kMxRing), (j / kMxRing) & 1, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never)) break;
    }
    if (lane == 0) {  // the x copy too (complete already unless a wait gave up)
      volatile int never = 0;
      mbar_wait(xbar, 0u, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never);
    }
  } else {
    const int grp = warp / kMxGW, wq = warp % kMxGW;
    const int g = lane >> 2, c = lane & 3;
    const int bar_grp = kMxBarGroup + grp;
    float *hf = p.ws.h;  // [k*K][I] fp32, by sorted pair position
    uint32_t range = 0;  // largest (scale - 113) met, unsigned
    bool dead = s_abort != 0;

    const int xrow = d * 2;  // bytes per staged x row
    const uint32_t xs = smem_u32(scratch);
    // the k rows of x (bf16, copied in at the start) become fp16 in place,
    // each times the power of two that puts its largest magnitude in
    // [2^14, 2^15) (warp t: row t).  The loops stay rolled: this code runs
    // once per launch, so its size (cold instruction fetch), not its
    // instruction count, sets its time.
    if (warp < k) {
      const int t = warp, cpr = d / 8;
      unsigned char *row = scratch + (size_t)t * xrow;
      const float inv = p.fuse_norm ? s_inv[t] : 1.f;
      // largest magnitude: bf16 patterns without the sign compare as integers
      uint32_t mb = 0;
#pragma unroll 1
      for (int q = lane; q < cpr; q += 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + q * 16);
        mb = __vmaxu2(mb, __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                   __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
      }
      mb = __reduce_max_sync(0xffffffffu, max(mb & 0xffffu, mb >> 16));
      float amax = __uint_as_float(mb << 16);
      if (p.fuse_norm) amax = rnd_bf16(amax * inv);  // rounding is monotone: the max of the rounded rows
      const int sh = row_shift(amax);
      const float sc = exp2i(sh);
#pragma unroll 1
      for (int q0 = 0; q0 < cpr; q0 += 32) {
        const int q = q0 + lane;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (q < cpr) v = *reinterpret_cast<const uint4 *>(row + q * 16);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float a = bf16_lo(w4[h]), b = bf16_hi(w4[h]);
          if (p.fuse_norm) {
            a = rnd_bf16(a * inv);
            b = rnd_bf16(b * inv);
          }
          o4[h] = pack_h2(a * sc, b * sc);
        }
        __syncwarp();  // the 32 chunks of this pass are read before any is rewritten
        if (q < cpr) *reinterpret_cast<uint4 *>(row + swz(q, t) * 16) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (lane == 0) s_xinv[t] = exp2i(-sh);
    }
    bar_sync_n(kBarAll, kFC);  // every staged x row is fp16 before any group reads it
    int cs = grp, cph = 0;  // ring slot and phase of this group's next stage
    auto stage_wait = [&]() {
      if (!dead && !mbar_wait_fast(full0 + 8 * cs, cph, p.ws.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) dead = true;
    };
    auto stage_release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * cs);
      cs += kMxGroups;
      if (cs >= kMxRing) {
        cs -= kMxRing;
        cph ^= 1;
      }
    };

    // ---------------------------------------------------------------- P2: gate/up
    // Token columns 0-7 accumulate in registers.  An expert with more than 8
    // tokens (k > 8 only) gets a second pass over the same stage for columns
    // 8-15: the codes are read again from the stage, which is released only
    // after that, and the sums of those columns live in shared memory between
    // stages.  Both passes add in the same order.
    const int rw = wq * 8 + g;  // this lane's row within the 32-row stage
    // B-row addresses of token column `n0 + g` of the expert at `off`
    auto x_rows = [&](int off, int m, int n0, uint32_t (&bt)[4]) {
      const int n = n0 + g;
      const int t = pair_token(s_gat[off + (n < m ? n : 0)], p.k, p.K);  // past m: any valid row, discarded
      const int sw = ((c >> 1) & 1) | ((t & 1) << 1);
      const uint32_t b0 = xs + t * xrow + c * 64;
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) bt[tt] = b0 + ((tt ^ sw) << 4);
    };
    auto g_load = [&](uint4 (&ag)[kMxCh], uint4 (&au)[kMxCh], uint32_t (&eg)[kMxCh], uint32_t (&eu)[kMxCh]) {
      const uint32_t st = sbase + cs * slot;
      const uint32_t ar = st + rw * (kMxCols / 2) + c * 16;
      const uint32_t sr = st + g_sc + rw * (kMxCols / 32) + c;
#pragma unroll
      for (int j = 0; j < kMxCh; ++j) {
        ag[j] = ld16(ar + j * 64);
        au[j] = ld16(ar + g_up + j * 64);
        eg[j] = ld1(sr + j * 4);
        eu[j] = ld1(sr + (g_scu - g_sc) + j * 4);
      }
    };
    auto g_mma = [&](float (&acc)[4], const uint4 (&ag)[kMxCh], const uint4 (&au)[kMxCh],
                     const uint32_t (&eg)[kMxCh], const uint32_t (&eu)[kMxCh], const uint32_t (&bt)[4], int q) {
#pragma unroll
      for (int j = 0; j < kMxCh; ++j) {
        const uint32_t sgv = e8m0_half2(eg[j], range), suv = e8m0_half2(eu[j], range);
        const int xo = (q * kMxCh + j) * 256;  // this chunk's bytes in a staged x row
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          uint32_t rg4[4], ru4[4];
          mx_decode_word(word_of(ag[j], tt), sgv, rg4);
          mx_decode_word(word_of(au[j], tt), suv, ru4);
          const uint4 b = ld16(bt[tt] + xo);
          mma_f16x(acc, rg4[0], ru4[0], rg4[1], ru4[1], b.x, b.y);
          mma_f16x(acc, rg4[2], ru4[2], rg4[3], ru4[3], b.z, b.w);
        }
      }
    };
    for (int r = 0; r < R2; ++r) {
      const int u = lo_g + r * kMxGroups + grp;
      const bool live = u < hi_g && !dead;
      int wi = 0, i0 = 0, off = 0, m = 0;
      uint32_t bt[4] = {0u, 0u, 0u, 0u};
      if (live) {
        wi = u / tiles_g;
        i0 = (u - wi * tiles_g) * kMxRows + wq * 8;
        off = s_off[wi];
        m = s_off[wi + 1] - off;
        x_rows(off, m, 0, bt);
      }
      const bool two = NT == 2 && live && m > 8;
      float *a1s = acc1s + (warp * 32 + lane) * 4;
      if (two) *reinterpret_cast<float4 *>(a1s) = make_float4(0.f, 0.f, 0.f, 0.f);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < nq; ++q) {
        stage_wait();
        if (!live || dead) {
          stage_release();
          continue;
        }
        uint4 ag[kMxCh], au[kMxCh];
        uint32_t eg[kMxCh], eu[kMxCh];
        g_load(ag, au, eg, eu);
        if (!two) stage_release();  // the codes are in registers: refill at once
        g_mma(acc, ag, au, eg, eu, bt, q);
        if (NT == 2 && two) {
          g_load(ag, au, eg, eu);
          stage_release();
          uint32_t bt1[4];
          x_rows(off, m, 8, bt1);
          const float4 v = *reinterpret_cast<const float4 *>(a1s);
          float a1[4] = {v.x, v.y, v.z, v.w};
          g_mma(a1, ag, au, eg, eu, bt1, q);
          *reinterpret_cast<float4 *>(a1s) = make_float4(a1[0], a1[1], a1[2], a1[3]);
        }
      }
      if (live && !dead) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = 2 * c + q;
          if (tok < m) {
            const float inv = s_xinv[pair_token(s_gat[off + tok], p.k, p.K)];
            hf[(size_t)(off + tok) * I + i0 + g] = silu(acc[q] * inv) * (acc[q + 2] * inv);
          }
        }
        if (NT == 2 && two) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int tok = 8 + 2 * c + q;
            if (tok < m) {
              const float inv = s_xinv[pair_token(s_gat[off + tok], p.k, p.K)];
              hf[(size_t)(off + tok) * I + i0 + g] = silu(a1s[q] * inv) * (a1s[q + 2] * inv);
            }
          }
        }
      }
    }
    // the staged x rows are dead once the CTA's gate/up work is done; publish
    // that (one release covers every h row this CTA wrote).  A down unit waits
    // only for the CTAs that own its expert's gate/up units.
    bar_sync_n(kBarAll, kFC);
    if (tid == 0) red_release_add(p.ws.flags + blockIdx.x, 1u);
    dead = dead || s_abort != 0;

    // ---------------------------------------------------------------- P3: down
    const int CI = (I + 127) / 128;
    const int hrow = CI * 256;  // bytes per staged h row
    unsigned char *hrows = scratch + (size_t)grp * (NT * 8) * hrow;
    const uint32_t hb = smem_u32(hrows);
    const bool tail_dead = (I & 127) != 0 && c >= 2;
    int cur = -1, m = 0, off = 0;
    for (int r = 0; r < R3; ++r) {
      const int u = lo_d + r * kMxGroups + grp;
      const bool live = u < hi_d;
      const int wi = live ? u / tiles_d : cur, dt = live ? u - wi * tiles_d : 0;
      if (live && wi != cur) {
        if (wq == 0 && !dead) {
          // gate/up unit u is CTA floor(((u + 1) G - 1) / U)'s
          const long long U = (long long)nW * tiles_g;
          const int b0 = (int)(((long long)(wi * tiles_g + 1) * G - 1) / U);
          const int b1 = (int)(((long long)((wi + 1) * tiles_g) * G - 1) / U);
          if (!ctas_done(p.ws.flags, b0, b1, p.ws.err, &s_abort)) dead = true;
        }
        bar_sync_n(bar_grp, kMxGW * 32);  // h of this expert complete; the previous one's rows are no longer read
        dead = dead || s_abort != 0;
        cur = wi;
        off = s_off[wi];
        m = s_off[wi + 1] - off;
        for (int n = wq; n < m; n += kMxGW) {
          const float *src = hf + (size_t)(off + n) * I;
          const int hcpr = I / 8;
          float4 v[2][2];
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int q = lane + 32 * i;
            v[i][0] = v[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q < hcpr) {
              v[i][0] = __ldcg(reinterpret_cast<const float4 *>(src + q * 8));
              v[i][1] = __ldcg(reinterpret_cast<const float4 *>(src + q * 8 + 4));
            }
            amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(v[i][0].x), fabsf(v[i][0].y)),
                                           fmaxf(fabsf(v[i][0].z), fabsf(v[i][0].w))),
                                     fmaxf(fmaxf(fabsf(v[i][1].x), fabsf(v[i][1].y)),
                                           fmaxf(fabsf(v[i][1].z), fabsf(v[i][1].w)))));
          }
          const int sh = row_shift(warp_max(amax));
          const float sc = exp2i(sh);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int q = lane + 32 * i;
            if (q < CI * 16)
              *reinterpret_cast<uint4 *>(hrows + (size_t)n * hrow + swz(q, n) * 16) =
                  make_uint4(pack_h2(v[i][0].x * sc, v[i][0].y * sc), pack_h2(v[i][0].z * sc, v[i][0].w * sc),
                             pack_h2(v[i][1].x * sc, v[i][1].y * sc), pack_h2(v[i][1].z * sc, v[i][1].w * sc));
          }
          if (lane == 0) s_hinv[grp][n] = exp2i(-sh);
        }
        bar_sync_n(bar_grp, kMxGW * 32);
      }
      stage_wait();
      if (!live || dead) {
        stage_release();
        continue;
      }
      const int r0 = dt * 64 + wq * 16;
      const bool two = NT == 2 && m > 8;
      uint4 a0[kMxCh], a1[kMxCh];
      uint32_t e0[kMxCh], e1[kMxCh];
      auto d_load = [&]() {
        const uint32_t st = sbase + cs * slot;
        const int rr = wq * 16 + g;
        const uint32_t ar = st + rr * rowb_d + c * 16;
        const uint32_t sr = st + d_sc + rr * srow_d + c;
#pragma unroll
        for (int j = 0; j < kMxCh; ++j) {
          a0[j] = a1[j] = make_uint4(0u, 0u, 0u, 0u);
          e0[j] = e1[j] = 127u;
          if (j < CI && !(tail_dead && j == CI - 1)) {
            a0[j] = ld16(ar + j * 64);
            a1[j] = ld16(ar + 8 * rowb_d + j * 64);
            e0[j] = ld1(sr + j * 4);
            e1[j] = ld1(sr + 8 * srow_d + j * 4);
          }
        }
      };
      // one pass = token columns n0..n0+7 of this expert over the stage's codes
      auto d_pass = [&](int n0) {
        uint32_t bt[4];
        {
          const int n = n0 + g, nn = n < m ? n : 0;
          const int sw = ((c >> 1) & 1) | ((nn & 1) << 1);
          const uint32_t b0 = hb + nn * hrow + c * 64;
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) bt[tt] = b0 + ((tt ^ sw) << 4);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kMxCh; ++j) {
          if (j < CI) {
            const uint32_t s0 = e8m0_half2(e0[j], range), s1 = e8m0_half2(e1[j], range);
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
              uint32_t r0v[4], r1v[4];
              mx_decode_word(word_of(a0[j], tt), s0, r0v);
              mx_decode_word(word_of(a1[j], tt), s1, r1v);
              const uint4 b = ld16(bt[tt] + j * 256);
              mma_f16x(acc, r0v[0], r1v[0], r0v[1], r1v[1], b.x, b.y);
              mma_f16x(acc, r0v[2], r1v[2], r0v[3], r1v[3], b.z, b.w);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = n0 + 2 * c + q;
          if (tok < m) {
            const int pair = s_gat[off + tok];
            const float w = s_w[pair] * s_hinv[grp][tok];
            p.ws.ys[(size_t)pair * d + r0 + g] = w * acc[q];
            p.ws.ys[(size_t)pair * d + r0 + g + 8] = w * acc[q + 2];
          }
        }
      };
      d_load();
      if (!two) stage_release();  // the codes are in registers: refill at once
      d_pass(0);
      if (NT == 2 && two) {  // an expert with more than 8 tokens: columns 8-15
        d_load();
        stage_release();
        d_pass(8);
      }
    }
    // ---- grid barrier 2: every ys row is written
    bar_sync_n(kBarAll, kFC);
    if (tid == 0 && !grid_sync(p, 2)) s_abort = 1;
    bar_sync_n(kBarAll, kFC);
    dead = dead || s_abort != 0;

    // ---------------------------------------------------------------- P4: combine
    if (!dead) {
      const int n_out = k * d;
      const int o0 = (int)(((long long)blockIdx.x * n_out) / G), o1 = (int)(((long long)(blockIdx.x + 1) * n_out) / G);
      for (int o = o0 + tid; o < o1; o += kFC) {
        const int t = o / d, rrow = o - t * d;
        float sum = 0.f;
        for (int sl = 0; sl < K; ++sl) sum += __ldcg(p.ws.ys + (size_t)(t * K + sl) * d + rrow);
        if (p.ns) sum += __ldcg(p.ws.ys + (size_t)(k * K + t) * d + rrow);  // shared expert
        if (p.residual) sum = load_act(p.residual, (size_t)t * d + rrow, DFV_BF16) + sum;
        store_act(p.out, (size_t)t * d + rrow, DFV_BF16, sum);
      }
    }
    if (range > kScaleRangeMax) atomicOr(p.ws.err, DFV_DEVERR_SCALE_RANGE);
  }

  // exit ticket: the last CTA out resets the grid-barrier count for the next launch
  __syncthreads();
  if (tid == 0) s_last_cta = atomicAdd(p.ws.sync + 1, 1u) == (unsigned)(G - 1);
  __syncthreads();
  if (s_last_cta) {
    __threadfence();
    for (int i = tid; i < G; i += blockDim.x) p.ws.flags[i] = 0u;
    if (tid == 0) {
      atomicExch(p.ws.sync, 0u);
      atomicExch(p.ws.sync + 1, 0u);
    }
  }
}

template <int NT>
size_t mx_smem(int d, int I, size_t *slot_out, size_t *scratch_out) {
  size_t gslot = (size_t)kMxRows * kMxCols + (size_t)kMxRows * kMxCols / 16, dslot = (size_t)34 * I;
  size_t slot = gslot > dslot ? gslot : dslot;
  slot = (slot + 127) & ~(size_t)127;
  const size_t ipad = (size_t)(I + 127) / 128 * 128;
  size_t xsb = (size_t)NT * 8 * d * 2, hsb = (size_t)kMxGroups * NT * 8 * ipad * 2;
  size_t scratch = xsb > hsb ? xsb : hsb;
  scratch = (scratch + 127) & ~(size_t)127;
  *slot_out = slot;
  *scratch_out = scratch;
  return (size_t)kMxRing * slot + scratch + 16 * kMxRing + (NT == 2 ? (size_t)kFW * 32 * 16 : 0);
}

}  // namespace
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char *why, size_t why_len);
namespace {

// 2-D uint8 tensor map over a [rows][cols] byte matrix with a box of bx x by.
bool encode_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by, char *why,
               size_t why_len) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, why_len);
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {bx, by};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(why, why_len, "mxfp4: tensor map encode failed (%d)", (int)r);
    return false;
  }
  return true;
}

}  // namespace

// ----------------------------------------------------------------------------
// host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char *why, size_t why_len) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(mu);
  if (!tried) {
    tried = true;
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  }
  if (!fn) snprintf(why, why_len, "mxfp4: cuTensorMapEncodeTiled is not available");
  return fn;
}

bool fused_mx_plan(int k, int d, int I, int E, FusedPlan *plan) {
  if (k < 1 || k > kMaxBlock || E < 1 || E > kMaxExperts) return false;
  if (d % kMxCols || d > kMxMaxD || I % 64 || I > 128 * kMxCh) return false;
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

bool fused_mx_tensor_maps(FusedParams *p, const dfv_moe_layer *L, char *why, size_t why_len) {
  // encoded maps are cached per (weights, shape): encoding is host work only
  struct Maps {
    CUtensorMap wg, wu, sg, su;
  };
  static std::mutex mu;
  static std::map<std::tuple<const void *, const void *, const void *, const void *, int, int, int>, Maps> cache;
  const auto key = std::make_tuple(L->w_gate, L->w_up, (const void *)L->s_gate, (const void *)L->s_up, L->d, L->d_ff,
                                   L->n_experts + (L->n_shared ? 1 : 0));
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      p->tm_wg = it->second.wg;
      p->tm_wu = it->second.wu;
      p->tm_sg = it->second.sg;
      p->tm_su = it->second.su;
      return true;
    }
  }
  Maps m;
  const uint64_t rows = (uint64_t)(L->n_experts + (L->n_shared ? 1 : 0)) * L->d_ff;  // the shared expert is the last
  if (!encode_2d(&m.wg, L->w_gate, L->d / 2, rows, kMxCols / 2, kMxRows, why, why_len) ||
      !encode_2d(&m.wu, L->w_up, L->d / 2, rows, kMxCols / 2, kMxRows, why, why_len) ||
      !encode_2d(&m.sg, L->s_gate, L->d / 32, rows, kMxCols / 32, kMxRows, why, why_len) ||
      !encode_2d(&m.su, L->s_up, L->d / 32, rows, kMxCols / 32, kMxRows, why, why_len))
    return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  p->tm_wg = m.wg;
  p->tm_wu = m.wu;
  p->tm_sg = m.sg;
  p->tm_su = m.su;
  return true;
}

// A cooperative launch (the grid barriers need every CTA resident), chained
// to the previous kernel programmatically when `pdl`: CTAs may start while it
// drains, and do nothing before griddepcontrol.wait.
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
  if (sms > 1024) {  // the per-CTA flags in the workspace hold 1024 CTAs
    snprintf(why, why_len, "mxfp4: %d SMs exceed the 1024 workspace flags", sms);
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
