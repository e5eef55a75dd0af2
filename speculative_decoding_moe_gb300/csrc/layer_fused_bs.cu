// layer_fused_bs.cu -- one MoE layer of a verify block in a single persistent,
// cooperative launch, with block-scaled expert weights: mxfp4 (E2M1 codes, one
// E8M0 power-of-two scale per 32 elements of a row) or 8-bit (int8 codes, one
// IEEE binary16 scale per 32 elements, llama.cpp's Q8_0 block); bf16 router and
// bf16 activations.
//
// "Speculating on a Strix Halo", sections "What the pieces cost" and "The
// verify's own cost": the block's tokens route to their own top-K experts, the
// block wakes their union, and tokens are grouped by expert.  The MI355X /
// vLLM write-up (allbreaknews.com/?p=4397), sections "Why Quantize the Target
// Model on Top?" and "Results: Quantizing the Target Model": the expert
// weights stay narrow all the way to the GEMM; "Speculating on a Strix Halo
// (part 2)", section "The verification cog": the target runs "at Q8".  Here
// each woken expert's codes and scales cross HBM exactly once and are widened
// to fp16 in registers.
//
// One CTA per SM: 16 consumer warps in 4 groups of 4, and one producer warp
// that streams the weights through an 8-stage mbarrier ring.  The producer
// feeds the groups round-robin, so group q consumes stages q, q+4, ... (a
// group with no unit left in a round gets an empty stage).
//
// Stage geometry, the same for both formats: 256 bytes of codes per weight row
// (512 mxfp4 codes or 256 8-bit codes) and the 16 bytes of scales that cover
// them.  Codes arrive as tensor-map boxes of 64 bytes x rows with the 64-byte
// swizzle, so that ldmatrix reads eight rows of a 16-byte chunk without bank
// conflicts; one 3-D copy brings the four boxes of a stage (the producer is a
// single thread, and one copy per box capped the stream rate).  ldmatrix hands
// lane (g, c) bytes 4c..4c+3 of each chunk of row g: for mxfp4 eight codes of
// one 32-element block, for 8-bit four codes of half a block.  Every MMA
// (m16n8k16, fp16 operands, fp32 accumulate; A = weights, B = tokens) therefore
// sums over the elements of one scale block only, and the block's scale
// multiplies the fp32 result: for every E8M0 exponent 0..254 and every binary16
// scale the products are exact, and only the fp32 sums round.  The token rows
// (x for gate/up, h for down) sit in shared memory as fp16, each multiplied by
// the power of two 2^sh that puts its largest magnitude in [1, 2), so the
// accumulators hold about the true sums (no overflow short of the fp32 range
// itself) and 2^-sh brings them back; bf16 elements down to 2^-17 of their
// row's largest stay exact, and smaller ones round at 2^-25 of it; for 8-bit
// weights the 32 elements of each block are stored in the order the MMA's k
// slots take them, so one 16-byte load feeds two MMAs in both formats.
//
//   P0, P1  routing, shared with the bf16 single-launch kernel (route_p0,
//       route_p1, on the k rows of x the producer copies into the staged-x
//       rows at the start; the producer starts streaming as soon as the woken
//       list is known).
//   P2  the k rows of x become fp16 in place while the first stages are in
//       flight.  unit = (woken expert, 32 d_ff rows), streamed as stages of 32
//       gate rows and 32 up rows; warp w of the group owns rows 8w..8w+7 over
//       the whole of d (gate rows = M 0-7, up rows = M 8-15, the expert's
//       tokens = N) and keeps its sums in registers across the stages;
//       h = silu(g) * u goes to global memory in fp32.  When all its gate/up
//       units are done, the CTA sets its own flag in the workspace.
//   P3  unit = (woken expert, 64 d rows), one or two stages of down codes.
//       Before it first reads an expert's h, a group waits (acquire, bounded)
//       for the flags of the CTAs that own that expert's gate/up units, then
//       stages the expert's h rows as fp16.  Each warp owns 16 rows.
//       w[t,s] * y goes to ys[pair].
//       -- grid barrier 2 --
//   P4  every CTA sums ys over the K slots in slot order (then the shared
//       slot) for its share of the output rows, adds the residual and writes
//       them.  The sum order of every output depends only on its own token.
// Every wait is bounded (2 s) and reports through the workspace error word.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "fused_common.cuh"
#include "mxfp4_common.cuh"

namespace dfv {
namespace {

constexpr int kBsGroups = 4;             // consumer groups
constexpr int kBsGW = kFW / kBsGroups;   // warps per group
constexpr int kBsRing = 8;               // ring stages (two per group)
constexpr int kBsBarGroup = 2;           // named barriers 2..5, one per group
constexpr int kBsRowsG = 32;             // d_ff rows per gate/up unit (8 per warp)
constexpr int kBsRowsD = 64;             // d rows per down unit (16 per warp)
constexpr int kBsRowBytes = 256;         // code bytes per row and stage
constexpr int kBsBox = 64;               // code box width in bytes (64-byte swizzle)
constexpr int kBsMaxD = 2048;            // staged x: k rows of d fp16 in 64 KB
constexpr uint32_t kBsCodes = 16384;     // code bytes of a stage (both layouts)
constexpr uint32_t kBsStage = 17408;     // + 1 KB of scales
constexpr uint32_t kBsSlot = 18432;      // slot stride, a multiple of 1024 (swizzle alignment)
constexpr int kFmtMx = 0, kFmtQ8 = 1;

// Format traits.  CPS: codes per row and stage; BPI: scale blocks per ldmatrix
// (four 16-byte chunks); SB: bytes per scale.
template <int FMT>
struct Fmt;
template <>
struct Fmt<kFmtMx> {
  static constexpr int CPS = 512, BPI = 4, SB = 1;
  // A fragments of block m of the four chunks ch[]: pairs of codes 8c..8c+7
  __device__ static __forceinline__ void frag(const uint32_t (&ch)[4], int m, uint32_t (&a)[4]) { e2m1_word(ch[m], a); }
  // the scale 2^(s-127) of block m of this iteration, from word `w` of the
  // row's scales: byte m moved into the fp32 exponent field (s = 0 gives
  // the fp32 subnormal 2^-127)
  __device__ static __forceinline__ float scale(uint32_t w, int m) {
    const uint32_t e = (m < 3 ? (w << (23 - 8 * m)) : (w >> 1)) & 0x7f800000u;
    return __uint_as_float(max(e, 0x00400000u));
  }
};
// int8 code bytes b0..b3 -> fp16x2 (b0, b1), (b2, b3), exactly: 0x64XX is
// 1024 + XX in fp16, XX = b + 128, and 1024 + 128 is subtracted.
__device__ __forceinline__ void q8_word(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5150), b = __byte_perm(u, 0x64646464u, 0x5352);
  const uint32_t bias = 0x64806480u;  // fp16x2 {1152, 1152}
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}
template <>
struct Fmt<kFmtQ8> {
  static constexpr int CPS = 256, BPI = 2, SB = 2;
  // block m = chunks 2m (codes 4c..4c+3: MMA 1) and 2m+1 (codes 16+4c..: MMA 2)
  __device__ static __forceinline__ void frag(const uint32_t (&ch)[4], int m, uint32_t (&a)[4]) {
    q8_word(ch[2 * m], a[0], a[1]);
    q8_word(ch[2 * m + 1], a[2], a[3]);
  }
  // block m's binary16 scale (exact in fp32)
  __device__ static __forceinline__ float scale(uint32_t w, int m) {
    return __half2float(__ushort_as_half((unsigned short)(m ? (w >> 16) : (w & 0xffffu))));
  }
};

// 16-byte chunk q of staged token row r sits at chunk q ^ ((r & 1) << 2):
// the quarter-warp reading chunks Q..Q+3 of rows 2i and 2i+1 then spans all
// 32 banks.
__device__ __forceinline__ int swz2(int q, int r) { return q ^ ((r & 1) << 2); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A * B (fp16, fp32 accumulate) from zero.
__device__ __forceinline__ void mma_f16_z(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Address of chunk j (0..3) of row `row` of a 64-byte-swizzled box at `box`.
__device__ __forceinline__ uint32_t sw64(uint32_t box, int row, int j) {
  return box + (uint32_t)row * kBsBox + ((uint32_t)(j ^ ((row >> 1) & 3)) << 4);
}

// 2-D tensor copy global -> shared with an L2 policy, x = innermost coordinate.
__device__ __forceinline__ void tma2(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar, uint64_t pol) {
  tma_2d_hint(dst, map, x, y, bar, pol);
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

// Stage the four 8-element chunks (w: this lane's chunk, fp16 pairs) of each
// 32-element block in the order the 8-bit MMA k slots take them: the lane
// holding chunk c' of a block ends up with elements 4c'..4c'+3 and
// 16+4c'..16+4c'+3.  The four lanes of a block are lanes 4i..4i+3.
__device__ __forceinline__ void q8_permute(uint32_t (&w)[4]) {
  const int lane = threadIdx.x & 31, cc = lane & 3, base = lane & ~3;
  const int s1 = base + (cc >> 1), s2 = base + 2 + (cc >> 1);
  uint32_t a[4], b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[i] = __shfl_sync(0xffffffffu, w[i], s1);
    b[i] = __shfl_sync(0xffffffffu, w[i], s2);
  }
  const bool h = cc & 1;
  w[0] = h ? a[2] : a[0];
  w[1] = h ? a[3] : a[1];
  w[2] = h ? b[2] : b[0];
  w[3] = h ? b[3] : b[1];
}

// NT: token tiles of 8 (k <= 8: 1); SINGLE: instantiated for k = 1 only.
template <int FMT, int NT, bool SINGLE>
__global__ void __launch_bounds__(kFT, 1) moe_fused_bs_kernel(const __grid_constant__ FusedParams p) {
  using F = Fmt<FMT>;
  pdl_trigger();
  prefetch_router_rows(p);
  pdl_wait();  // before this only the router-row prefetch touches global memory
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled boxes need 1024-byte aligned slots
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = p.k, d = p.d, I = p.I, K = p.K;
  const int G = gridDim.x;
  const uint32_t sbase = smem_u32(smem);
  unsigned char *scratch = smem + kBsRing * kBsSlot;  // x rows (P2), h rows per group (P3)
  const uint32_t full0 = sbase + kBsRing * kBsSlot + p.scratch;
  const uint32_t empty0 = full0 + 8 * kBsRing;

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
  __shared__ float s_hinv[kBsGroups][kMaxBlock];  // 2^-shift of each staged h row, per group
  __shared__ int s_nw;
  __shared__ unsigned s_last_cta;
  __shared__ volatile int s_abort, s_bad;
  __shared__ __align__(8) unsigned long long s_xbar;  // the copy of the k rows of x

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t xbar = smem_u32(&s_xbar);
  if (tid == 0) {
    s_abort = 0;
    s_bad = 0;
    for (int s = 0; s < kBsRing; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kBsGW);
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
    prefetch_tensormap(&p.tm_wd);
  }
  if (consumer) {
    const RouteSmem rs = {s_idx, s_w, s_woken, s_off, s_eoff, s_gat, s_tmask, s_inv, &s_nw, &s_abort, &s_bad};
    const RouteArgs ra = route_args(p, rs, reinterpret_cast<const uint16_t *>(scratch), xbar);
    route_p0(ra);
    route_p1<SINGLE>(ra, [](int) {});
  } else {
    bar_sync_n(kBarProducer, 64);  // released as soon as the woken list is known
  }

  const int nW = s_nw;  // 0 when the CTA aborted before its routing
  const int tiles_g = I / kBsRowsG, tiles_d = d / kBsRowsD;
  const int nq = d / F::CPS;                       // gate/up stages per unit
  const int rowb_d = I * (FMT == kFmtMx ? 1 : 2) / 2;  // down code bytes per row
  const int nqd = (rowb_d + kBsRowBytes - 1) / kBsRowBytes;  // down stages per unit
  const int srow_d = I / 32 * F::SB;                // down scale bytes per row
  const int srs_d = nqd == 1 ? srow_d : 16;         // ... per row and stage, as staged
  int lo_g, hi_g, lo_d, hi_d;
  {
    const int U = nW * tiles_g, V = nW * tiles_d;
    lo_g = (int)((unsigned)blockIdx.x * (unsigned)U / (unsigned)G);
    hi_g = (int)((unsigned)(blockIdx.x + 1) * (unsigned)U / (unsigned)G);
    lo_d = (int)((unsigned)blockIdx.x * (unsigned)V / (unsigned)G);
    hi_d = (int)((unsigned)(blockIdx.x + 1) * (unsigned)V / (unsigned)G);
  }
  const int R2 = (hi_g - lo_g + kBsGroups - 1) / kBsGroups, R3 = (hi_d - lo_d + kBsGroups - 1) / kBsGroups;
  // gate/up stage: [4 boxes][32 rows][64 B] gate | the same for up |
  // [32][16] gate scales | [32][16] up scales.  down stage: [<= 4 boxes][64
  // rows][64 B] codes | [64][srs_d] scales
  constexpr uint32_t kUpOff = kBsCodes / 2, kScOff = kBsCodes, kScUpOff = kBsCodes + 512;

  if (!consumer) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && !s_abort) {
      const uint64_t pol = l2_evict_first();  // expert weights are read once per launch
      int it = 0, ps = 0, pph = 0;            // stages issued; slot and phase of the next one
      bool ok = true;
      auto take = [&]() -> bool {
        return mbar_wait_fast(empty0 + 8 * ps, pph ^ 1, p.ws.err, DFV_DEVERR_SLOT_WAIT, &s_abort);
      };
      auto advance = [&]() {
        ++it;
        if (++ps == kBsRing) {
          ps = 0;
          pph ^= 1;
        }
      };
      // gate/up: rounds of one unit per group, nq stages per unit
      for (int r = 0; r < R2 && ok; ++r) {
        for (int q = 0; q < nq && ok; ++q) {
          for (int gq = 0; gq < kBsGroups; ++gq) {
            if (!take()) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * kBsSlot;
            const int u = lo_g + r * kBsGroups + gq;
            if (u < hi_g) {
              const int wi = u / tiles_g;
              const int row = s_woken[wi] * I + (u - wi * tiles_g) * kBsRowsG;
              mbar_expect_tx(fb, kBsStage);
              // the stage's four 64-byte boxes of 32 rows in one copy each
              tma_3d_hint(dst, &p.tm_wg, 0, row, q * 4, fb, pol);
              tma_3d_hint(dst + kUpOff, &p.tm_wu, 0, row, q * 4, fb, pol);
              tma2(dst + kScOff, &p.tm_sg, q * 16, row, fb, pol);
              tma2(dst + kScUpOff, &p.tm_su, q * 16, row, fb, pol);
            } else {
              mbar_arrive(fb);  // empty stage: this group has no unit in this round
            }
            advance();
          }
        }
      }
      // down: rounds of one unit per group, nqd stages per unit
      for (int r = 0; r < R3 && ok; ++r) {
        for (int q = 0; q < nqd && ok; ++q) {
          for (int gq = 0; gq < kBsGroups; ++gq) {
            if (!take()) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8 * ps, dst = sbase + ps * kBsSlot;
            const int u = lo_d + r * kBsGroups + gq;
            if (u < hi_d) {
              const int wi = u / tiles_d;
              const int row = s_woken[wi] * d + (u - wi * tiles_d) * kBsRowsD;
              // one copy of the stage's min(4, boxes per row) boxes (the shapes
              // the plan takes have no partial last stage)
              const int bz = min(4, rowb_d / kBsBox);
              mbar_expect_tx(fb, (uint32_t)(bz * kBsRowsD * kBsBox + kBsRowsD * srs_d));
              tma_3d_hint(dst, &p.tm_wd, 0, row, q * 4, fb, pol);
              if (nqd == 1)
                bulk_g2s_hint(dst + kScOff, p.sd + (size_t)row * srow_d, (uint32_t)(kBsRowsD * srow_d), fb, pol);
              else
                tma2(dst + kScOff, &p.tm_sd, q * 16, row, fb, pol);
            } else {
              mbar_arrive(fb);
            }
            advance();
          }
        }
      }
      // no copy may land after the CTA exits
      volatile int never = 0;
      for (int j = it - kBsRing < 0 ? 0 : it - kBsRing; j < it; ++j)
        if (!mbar_wait(full0 + 8 * (j % kBsRing), (j / kBsRing) & 1, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never)) break;
    }
    if (lane == 0) {  // the x copy too (complete already unless a wait gave up)
      volatile int never = 0;
      mbar_wait(xbar, 0u, p.ws.err, DFV_DEVERR_DRAIN_WAIT, &never);
    }
  } else {
    const int grp = warp / kBsGW, wq = warp % kBsGW;
    const int g = lane >> 2, c = lane & 3;
    const int bar_grp = kBsBarGroup + grp;
    float *hf = p.ws.h;  // [k*K][I] fp32, by sorted pair position
    bool dead = s_abort != 0;
    const int xrow = d * 2;  // bytes per staged x row
    const uint32_t xs = smem_u32(scratch);

    // the k rows of x (bf16, copied in at the start) become fp16 in place,
    // each times the power of two that puts its largest magnitude in [1, 2)
    // (warp t: row t), chunks swizzled (and, for 8-bit weights,
    // each block's elements in k-slot order).  The loops stay rolled: this
    // code runs once per launch, so its size (cold instruction fetch), not
    // its instruction count, sets its time.
    if (warp < k) {
      const int t = warp, cpr = d / 8;
      unsigned char *row = scratch + (size_t)t * xrow;
      const float inv = p.fuse_norm ? s_inv[t] : 1.f;
      uint32_t mb = 0;  // largest magnitude: bf16 patterns without the sign compare as integers
#pragma unroll 1
      for (int q = lane; q < cpr; q += 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + q * 16);
        mb = __vmaxu2(mb, __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                   __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
      }
      mb = __reduce_max_sync(0xffffffffu, max(mb & 0xffffu, mb >> 16));
      float amax = __uint_as_float(mb << 16);
      if (p.fuse_norm) amax = rnd_bf16(amax * inv);  // rounding is monotone: the max of the rounded row
      const int sh = row_shift(amax);
      const float sc = exp2i(sh);
#pragma unroll 1
      for (int q0 = 0; q0 < cpr; q0 += 32) {  // cpr is a multiple of 64
        const int q = q0 + lane;
        const uint4 v = *reinterpret_cast<const uint4 *>(row + q * 16);
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
        if (FMT == kFmtQ8) q8_permute(o4);
        __syncwarp();  // the 32 chunks of this pass are read before any is rewritten
        *reinterpret_cast<uint4 *>(row + swz2(q, t) * 16) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
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
      cs += kBsGroups;
      if (cs >= kBsRing) {
        cs -= kBsRing;
        cph ^= 1;
      }
    };
    // ldmatrix row of this lane: lane i supplies row (i & 7) of chunk (i >> 3)
    const int lrow = lane & 7, lchunk = lane >> 3;

    // ---------------------------------------------------------------- P2: gate/up
    // Tokens 0-7 (tile 0) and, for an expert with more than 8 tokens (k > 8
    // only), tokens 8-15 (tile 1) accumulate in registers over the stages.
    for (int r = 0; r < R2; ++r) {
      const int u = lo_g + r * kBsGroups + grp;
      const bool live = u < hi_g && !dead;
      int wi = 0, i0 = 0, off = 0, m = 0;
      uint32_t xb0 = 0, xb1 = 0;  // staged x rows of token columns g and 8 + g
      int t0 = 0, t1 = 0;
      if (live) {
        wi = u / tiles_g;
        i0 = (u - wi * tiles_g) * kBsRowsG + wq * 8;
        off = s_off[wi];
        m = s_off[wi + 1] - off;
        // past m: any valid row, its columns are discarded
        t0 = pair_token(s_gat[off + (g < m ? g : 0)], k, K);
        t1 = pair_token(s_gat[off + (8 + g < m ? 8 + g : 0)], k, K);
        xb0 = xs + t0 * xrow;
        xb1 = xs + t1 * xrow;
      }
      const bool two = NT == 2 && live && m > 8;
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int q = 0; q < nq; ++q) {
        stage_wait();
        if (!live || dead) {
          stage_release();
          continue;
        }
        const uint32_t st = sbase + cs * kBsSlot;
        const int rw = wq * 8 + g;  // this lane's gate / up row in the stage
        const uint4 sgv = lds128(st + kScOff + rw * 16), suv = lds128(st + kScUpOff + rw * 16);
        // B chunks: lane c's chunk of block blk of this stage in token row t
        // sits at 4 * (blk ^ (t & 1)) + c (swizzle): per parity, one base for
        // even and one for odd blocks, plus an immediate per block
        const uint32_t xq0 = (uint32_t)(q * (F::CPS / 8) + c) * 16;
        const uint32_t x0e = xb0 + xq0 + ((t0 & 1) ? 64u : 0u), x0o = xb0 + xq0 - ((t0 & 1) ? 64u : 0u);
        const uint32_t x1e = xb1 + xq0 + ((t1 & 1) ? 64u : 0u), x1o = xb1 + xq0 - ((t1 & 1) ? 64u : 0u);
        // unrolled by two: the next box's ldmatrix overlaps this box's MMAs
#pragma unroll 2
        for (int itb = 0; itb < 4; ++itb) {  // one box = four 16-byte chunks per row
          uint32_t cg[4], cu[4];
          ldsm_x4(sw64(st + itb * (kBsRowsG * kBsBox), wq * 8 + lrow, lchunk), cg);
          ldsm_x4(sw64(st + kUpOff + itb * (kBsRowsG * kBsBox), wq * 8 + lrow, lchunk), cu);
          const uint32_t swg = itb == 0 ? sgv.x : itb == 1 ? sgv.y : itb == 2 ? sgv.z : sgv.w;
          const uint32_t swu = itb == 0 ? suv.x : itb == 1 ? suv.y : itb == 2 ? suv.z : suv.w;
          const uint32_t ib = (uint32_t)itb * F::BPI * 64;
#pragma unroll
          for (int mb = 0; mb < F::BPI; ++mb) {
            uint32_t ag[4], au[4];
            F::frag(cg, mb, ag);
            F::frag(cu, mb, au);
            const float fg = F::scale(swg, mb), fu = F::scale(swu, mb);
            float tmp[4];
            {
              const uint4 b = lds128(((mb & 1) ? x0o : x0e) + ib + mb * 64);
              float tmp2[4];  // the block's two MMAs are independent: no MMA-to-MMA latency
              mma_f16_z(tmp, ag[0], au[0], ag[1], au[1], b.x, b.y);
              mma_f16_z(tmp2, ag[2], au[2], ag[3], au[3], b.z, b.w);
              acc0[0] = fmaf(fg, tmp[0] + tmp2[0], acc0[0]);
              acc0[1] = fmaf(fg, tmp[1] + tmp2[1], acc0[1]);
              acc0[2] = fmaf(fu, tmp[2] + tmp2[2], acc0[2]);
              acc0[3] = fmaf(fu, tmp[3] + tmp2[3], acc0[3]);
            }
            if (NT == 2 && two) {
              const uint4 b = lds128(((mb & 1) ? x1o : x1e) + ib + mb * 64);
              float tmp2[4];  // the block's two MMAs are independent: no MMA-to-MMA latency
              mma_f16_z(tmp, ag[0], au[0], ag[1], au[1], b.x, b.y);
              mma_f16_z(tmp2, ag[2], au[2], ag[3], au[3], b.z, b.w);
              acc1[0] = fmaf(fg, tmp[0] + tmp2[0], acc1[0]);
              acc1[1] = fmaf(fg, tmp[1] + tmp2[1], acc1[1]);
              acc1[2] = fmaf(fu, tmp[2] + tmp2[2], acc1[2]);
              acc1[3] = fmaf(fu, tmp[3] + tmp2[3], acc1[3]);
            }
          }
        }
        stage_release();
      }
      if (live && !dead) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = 2 * c + q;
          if (tok < m) {
            const float inv = s_xinv[pair_token(s_gat[off + tok], k, K)];
            hf[(size_t)(off + tok) * I + i0 + g] = silu(acc0[q] * inv) * (acc0[q + 2] * inv);
          }
          if (NT == 2 && two) {
            const int tok1 = 8 + 2 * c + q;
            if (tok1 < m) {
              const float inv = s_xinv[pair_token(s_gat[off + tok1], k, K)];
              hf[(size_t)(off + tok1) * I + i0 + g] = silu(acc1[q] * inv) * (acc1[q + 2] * inv);
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
    const int hrow = I * 2;  // bytes per staged h row (fp16)
    const int hcpr = I / 8;  // 16-byte chunks per h row
    unsigned char *hrows = scratch + (size_t)grp * (NT * 8) * hrow;
    const uint32_t hb = smem_u32(hrows);
    int cur = -1, m = 0, off = 0;
    for (int r = 0; r < R3; ++r) {
      const int u = lo_d + r * kBsGroups + grp;
      const bool live = u < hi_d;
      const int wi = live ? u / tiles_d : cur, dt = live ? u - wi * tiles_d : 0;
      if (live && wi != cur) {
        if (wq == 0 && !dead) {
          // gate/up unit u is CTA floor(((u + 1) G - 1) / U)'s
          const unsigned U = (unsigned)nW * tiles_g;
          const int b0 = (int)(((unsigned)(wi * tiles_g + 1) * (unsigned)G - 1u) / U);
          const int b1 = (int)(((unsigned)((wi + 1) * tiles_g) * (unsigned)G - 1u) / U);
          if (!ctas_done(p.ws.flags, b0, b1, p.ws.err, &s_abort)) dead = true;
        }
        bar_sync_n(bar_grp, kBsGW * 32);  // h of this expert complete; the previous one's rows are no longer read
        dead = dead || s_abort != 0;
        cur = wi;
        off = s_off[wi];
        m = s_off[wi + 1] - off;
        // this warp's rows n = wq, wq + 4, ... (at most NT * 2), two at a
        // time with all their loads in flight.  Lane l makes chunks l and
        // l + 32 (8 elements each) of a row.
#pragma unroll 1
        for (int n0 = wq; n0 < m; n0 += 2 * kBsGW) {
          const int nr = (n0 + kBsGW < m) ? 2 : 1;
          float4 v[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float4 *src = reinterpret_cast<const float4 *>(hf + (size_t)(off + n0 + j * kBsGW) * I);
#pragma unroll
            for (int cq = 0; cq < 2; ++cq) {
              const int q = lane + 32 * cq;
              const bool ok = j < nr && q < hcpr;
              v[j][2 * cq] = ok ? __ldcg(src + 2 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
              v[j][2 * cq + 1] = ok ? __ldcg(src + 2 * q + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j < nr) {
              const int n = n0 + j * kBsGW;
              float amax = 0.f;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j][i].x), fabsf(v[j][i].y)),
                                         fmaxf(fabsf(v[j][i].z), fabsf(v[j][i].w))));
              const int sh = row_shift(warp_max(amax));
              const float sc = exp2i(sh);
#pragma unroll
              for (int cq = 0; cq < 2; ++cq) {
                const int q = lane + 32 * cq;
                const float4 a = v[j][2 * cq], b = v[j][2 * cq + 1];
                uint32_t o4[4] = {pack_h2(a.x * sc, a.y * sc), pack_h2(a.z * sc, a.w * sc), pack_h2(b.x * sc, b.y * sc),
                                  pack_h2(b.z * sc, b.w * sc)};
                if (FMT == kFmtQ8) q8_permute(o4);
                if (q < hcpr)
                  *reinterpret_cast<uint4 *>(hrows + (size_t)n * hrow + swz2(q, n) * 16) =
                      make_uint4(o4[0], o4[1], o4[2], o4[3]);
              }
              if (lane == 0) s_hinv[grp][n] = exp2i(-sh);
            }
          }
        }
        bar_sync_n(bar_grp, kBsGW * 32);
      }
      const int r0 = dt * kBsRowsD + wq * 16;
      const bool two = NT == 2 && m > 8;
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t hb0 = hb + (uint32_t)(g < m ? g : 0) * hrow;
      const uint32_t hb1 = hb + (uint32_t)(8 + g < m ? 8 + g : 0) * hrow;
      const int n0s = g < m ? g : 0, n1s = 8 + g < m ? 8 + g : 0;
#pragma unroll 1
      for (int q = 0; q < nqd; ++q) {
        stage_wait();
        if (!live || dead) {
          stage_release();
          continue;
        }
        const uint32_t st = sbase + cs * kBsSlot;
        const int nb = min(4, (rowb_d - q * kBsRowBytes) / kBsBox);
        const int rlo = wq * 16 + g, rhi = rlo + 8;  // this lane's two rows in the stage
        const uint32_t hq0 = (uint32_t)(q * (F::CPS / 8) + c) * 16;
        const uint32_t h0e = hb0 + hq0 + ((n0s & 1) ? 64u : 0u), h0o = hb0 + hq0 - ((n0s & 1) ? 64u : 0u);
        const uint32_t h1e = hb1 + hq0 + ((n1s & 1) ? 64u : 0u), h1o = hb1 + hq0 - ((n1s & 1) ? 64u : 0u);
#pragma unroll 1
        for (int itb = 0; itb < nb; ++itb) {
          uint32_t c0r[4], c1r[4], wlo, whi;
          const uint32_t box = st + itb * (kBsRowsD * kBsBox);
          ldsm_x4(sw64(box, wq * 16 + lrow, lchunk), c0r);
          ldsm_x4(sw64(box, wq * 16 + 8 + lrow, lchunk), c1r);
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wlo) : "r"(st + kScOff + rlo * srs_d + itb * 4));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(whi) : "r"(st + kScOff + rhi * srs_d + itb * 4));
          const uint32_t ib = (uint32_t)itb * F::BPI * 64;
#pragma unroll
          for (int mb = 0; mb < F::BPI; ++mb) {
            uint32_t a0[4], a1[4];
            F::frag(c0r, mb, a0);
            F::frag(c1r, mb, a1);
            const float f0 = F::scale(wlo, mb), f1 = F::scale(whi, mb);
            float tmp[4];
            {
              const uint4 b = lds128(((mb & 1) ? h0o : h0e) + ib + mb * 64);
              float tmp2[4];  // the block's two MMAs are independent: no MMA-to-MMA latency
              mma_f16_z(tmp, a0[0], a1[0], a0[1], a1[1], b.x, b.y);
              mma_f16_z(tmp2, a0[2], a1[2], a0[3], a1[3], b.z, b.w);
              acc0[0] = fmaf(f0, tmp[0] + tmp2[0], acc0[0]);
              acc0[1] = fmaf(f0, tmp[1] + tmp2[1], acc0[1]);
              acc0[2] = fmaf(f1, tmp[2] + tmp2[2], acc0[2]);
              acc0[3] = fmaf(f1, tmp[3] + tmp2[3], acc0[3]);
            }
            if (NT == 2 && two) {
              const uint4 b = lds128(((mb & 1) ? h1o : h1e) + ib + mb * 64);
              float tmp2[4];  // the block's two MMAs are independent: no MMA-to-MMA latency
              mma_f16_z(tmp, a0[0], a1[0], a0[1], a1[1], b.x, b.y);
              mma_f16_z(tmp2, a0[2], a1[2], a0[3], a1[3], b.z, b.w);
              acc1[0] = fmaf(f0, tmp[0] + tmp2[0], acc1[0]);
              acc1[1] = fmaf(f0, tmp[1] + tmp2[1], acc1[1]);
              acc1[2] = fmaf(f1, tmp[2] + tmp2[2], acc1[2]);
              acc1[3] = fmaf(f1, tmp[3] + tmp2[3], acc1[3]);
            }
          }
        }
        stage_release();
      }
      if (live && !dead) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = 2 * c + q;
          if (tok < m) {
            const int pair = s_gat[off + tok];
            const float w = s_w[pair] * s_hinv[grp][tok];
            p.ws.ys[(size_t)pair * d + r0 + g] = w * acc0[q];
            p.ws.ys[(size_t)pair * d + r0 + g + 8] = w * acc0[q + 2];
          }
          if (NT == 2 && two) {
            const int tok1 = 8 + 2 * c + q;
            if (tok1 < m) {
              const int pair = s_gat[off + tok1];
              const float w = s_w[pair] * s_hinv[grp][tok1];
              p.ws.ys[(size_t)pair * d + r0 + g] = w * acc1[q];
              p.ws.ys[(size_t)pair * d + r0 + g + 8] = w * acc1[q + 2];
            }
          }
        }
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
      const int o0 = (int)((unsigned)blockIdx.x * (unsigned)n_out / (unsigned)G);
      const int o1 = (int)((unsigned)(blockIdx.x + 1) * (unsigned)n_out / (unsigned)G);
      for (int o = o0 + tid; o < o1; o += kFC) {
        const int t = o / d, rrow = o - t * d;
        float sum = 0.f;
        for (int sl = 0; sl < K; ++sl) sum += __ldcg(p.ws.ys + (size_t)(t * K + sl) * d + rrow);
        if (p.ns) sum += __ldcg(p.ws.ys + (size_t)(k * K + t) * d + rrow);  // shared expert
        if (p.residual) sum = load_act(p.residual, (size_t)t * d + rrow, DFV_BF16) + sum;
        store_act(p.out, (size_t)t * d + rrow, DFV_BF16, sum);
      }
    }
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

}  // namespace
}  // namespace dfv

// ----------------------------------------------------------------------------
// host side
namespace dfv {
namespace {

// shared memory of a launch: 1 KB of alignment slack | ring | staged x / h rows
// | full and empty mbarriers
template <int NT>
size_t bs_smem(int d, int I, size_t *scratch_out) {
  const size_t xsb = (size_t)NT * 8 * d * 2, hsb = (size_t)kBsGroups * NT * 8 * I * 2;
  size_t scratch = xsb > hsb ? xsb : hsb;
  scratch = (scratch + 127) & ~(size_t)127;
  *scratch_out = scratch;
  return 1024 + (size_t)kBsRing * kBsSlot + scratch + 16 * kBsRing;
}

template <int FMT>
void *bs_kernel(int k) {
  return k == 1   ? reinterpret_cast<void *>(moe_fused_bs_kernel<FMT, 1, true>)
         : k <= 8 ? reinterpret_cast<void *>(moe_fused_bs_kernel<FMT, 1, false>)
                  : reinterpret_cast<void *>(moe_fused_bs_kernel<FMT, 2, false>);
}
void *bs_kernel(int fmt, int k) { return fmt == DFV_Q8 ? bs_kernel<kFmtQ8>(k) : bs_kernel<kFmtMx>(k); }

// 2-D uint8 tensor map over a [rows][cols] byte matrix with a box of bx x by.
bool encode_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by,
               CUtensorMapSwizzle swizzle, char *why, size_t why_len);

}  // namespace

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
  if (!fn) snprintf(why, why_len, "block-scaled: cuTensorMapEncodeTiled is not available");
  return fn;
}

namespace {
// 3-D uint8 map over [rows][cols] bytes seen as [cols / 64][rows][64]: one box
// is min(4, cols / 64) consecutive 64-byte chunks of `by` rows, landing as
// that many [by][64] boxes with the 64-byte swizzle.
bool encode_3d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t by, char *why,
               size_t why_len) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, why_len);
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols, 64};
  const cuuint32_t box[3] = {64, by, (cuuint32_t)(cols / 64 < 4 ? cols / 64 : 4)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(why, why_len, "block-scaled: tensor map encode failed (%d)", (int)r);
    return false;
  }
  return true;
}

bool encode_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by,
               CUtensorMapSwizzle swizzle, char *why, size_t why_len) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, why_len);
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {bx, by};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(why, why_len, "block-scaled: tensor map encode failed (%d)", (int)r);
    return false;
  }
  return true;
}
}  // namespace

bool fused_bs_plan(int fmt, int k, int d, int I, int E, FusedPlan *plan) {
  if (k < 1 || k > kMaxBlock || E < 1 || E > kMaxExperts || d > kBsMaxD || I > 512 || I < 64) return false;
  if (fmt == DFV_MXFP4) {
    if (d % Fmt<kFmtMx>::CPS || I % 128) return false;
  } else if (fmt == DFV_Q8) {
    // a down row of more than one stage takes its scales in 16-byte boxes:
    // whole rows of scales then need a 16-byte multiple
    if (d % Fmt<kFmtQ8>::CPS || I % 64 || (I > 256 && I % 256)) return false;
  } else {
    return false;
  }
  size_t scratch = 0;
  const size_t smem = k <= 8 ? bs_smem<1>(d, I, &scratch) : bs_smem<2>(d, I, &scratch);
  if (smem + 8 * 1024 > 227 * 1024) return false;  // + the static shared memory (7 KB)
  plan->ks = 0;
  plan->nsl = 0;
  plan->slot = (int)kBsSlot;
  plan->scratch = (int)scratch;
  plan->ring = kBsRing;
  plan->smem = smem;
  return true;
}

bool fused_bs_tensor_maps(FusedParams *p, const dfv_moe_layer *L, char *why, size_t why_len) {
  // encoded maps are cached per (weights, shape): encoding is host work only
  struct Maps {
    CUtensorMap wg, wu, sg, su, wd, sd;
  };
  static std::mutex mu;
  static std::map<std::tuple<const void *, const void *, const void *, const void *, const void *, const void *, int,
                             int, int, int>,
                  Maps>
      cache;
  const int Et = L->n_experts + (L->n_shared ? 1 : 0);  // the shared expert is the last
  const auto key = std::make_tuple(L->w_gate, L->w_up, (const void *)L->s_gate, (const void *)L->s_up, L->w_down,
                                   (const void *)L->s_down, L->d, L->d_ff, Et, L->w_dtype);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      p->tm_wg = it->second.wg;
      p->tm_wu = it->second.wu;
      p->tm_sg = it->second.sg;
      p->tm_su = it->second.su;
      p->tm_wd = it->second.wd;
      p->tm_sd = it->second.sd;
      return true;
    }
  }
  const bool q8 = L->w_dtype == DFV_Q8;
  const uint64_t cbn = q8 ? 1 : 1, cbd = q8 ? 1 : 2;  // code bytes = elements * cbn / cbd
  const uint64_t sb = q8 ? 2 : 1;                      // bytes per scale
  const uint64_t d = L->d, I = L->d_ff;
  const uint64_t rows_g = (uint64_t)Et * I, rows_d = (uint64_t)Et * d;
  Maps m;
  memset(&m, 0, sizeof m);
  const bool multi = I * cbn / cbd > (uint64_t)kBsRowBytes;  // down rows of more than one stage
  if (!encode_3d(&m.wg, L->w_gate, d * cbn / cbd, rows_g, kBsRowsG, why, why_len) ||
      !encode_3d(&m.wu, L->w_up, d * cbn / cbd, rows_g, kBsRowsG, why, why_len) ||
      !encode_2d(&m.sg, L->s_gate, d / 32 * sb, rows_g, 16, kBsRowsG, CU_TENSOR_MAP_SWIZZLE_NONE, why, why_len) ||
      !encode_2d(&m.su, L->s_up, d / 32 * sb, rows_g, 16, kBsRowsG, CU_TENSOR_MAP_SWIZZLE_NONE, why, why_len) ||
      !encode_3d(&m.wd, L->w_down, I * cbn / cbd, rows_d, kBsRowsD, why, why_len) ||
      (multi &&
       !encode_2d(&m.sd, L->s_down, I / 32 * sb, rows_d, 16, kBsRowsD, CU_TENSOR_MAP_SWIZZLE_NONE, why, why_len)))
    return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  p->tm_wg = m.wg;
  p->tm_wu = m.wu;
  p->tm_sg = m.sg;
  p->tm_su = m.su;
  p->tm_wd = m.wd;
  p->tm_sd = m.sd;
  return true;
}

// A cooperative launch (the grid barriers need every CTA resident), chained
// to the previous kernel programmatically when `pdl`: CTAs may start while it
// drains, and do nothing before griddepcontrol.wait.
cudaError_t launch_fused_bs(const FusedParams &p0, int fmt, const FusedPlan &plan, int grid, cudaStream_t s,
                            bool pdl) {
  FusedParams p = p0;
  p.slot = plan.slot;
  p.scratch = plan.scratch;
  p.ring = plan.ring;
  void *kern = bs_kernel(fmt, p.k);
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
  void *args[] = {&p};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

int fused_bs_max_grid(const FusedPlan &plan, int fmt, int k, char *why, size_t why_len) {
  int dev = 0, sms = 0, per = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    snprintf(why, why_len, "SM count query: %s", cudaGetErrorString(e));
    return 0;
  }
  if (sms > 1024) {  // the per-CTA flags in the workspace hold 1024 CTAs
    snprintf(why, why_len, "block-scaled: %d SMs exceed the 1024 workspace flags", sms);
    return 0;
  }
  void *kern = bs_kernel(fmt, k);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(why, why_len, "block-scaled: shared memory %zu B: %s", plan.smem, cudaGetErrorString(e));
    return 0;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, kFT, plan.smem);
  if (e != cudaSuccess || per < 1) {
    cudaGetLastError();
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, kern);
    snprintf(why, why_len, "block-scaled: occupancy %d (%s): regs %d, static smem %zu, max threads %d, dyn smem %zu",
             per, cudaGetErrorString(e), fa.numRegs, fa.sharedSizeBytes, fa.maxThreadsPerBlock, plan.smem);
    return 0;
  }
  return sms;
}

}  // namespace dfv
