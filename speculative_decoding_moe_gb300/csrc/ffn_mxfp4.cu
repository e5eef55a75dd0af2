// ffn_mxfp4.cu -- grouped SwiGLU expert FFN and routing-weighted combine over
// experts stored in mxfp4: E2M1 codes, two per byte (low nibble = even column),
// with one E8M0 power-of-two scale per 32 consecutive elements of a row.
//
// The MI355X / vLLM write-up (allbreaknews.com/?p=4397), sections "Why Quantize
// the Target Model on Top?" and "Results: Quantizing the Target Model": the
// target's expert weights stay in fp4 and feed a native fp4 MoE kernel;
// widening them to bf16 in memory first would stream the wide expert stack
// every step and give the gain back.  Here every byte of codes and scales is
// read from HBM exactly once and widened in registers right before the MMA.
//
// Decode.  A quad's four lanes (c = 0..3) read 64 contiguous bytes of a row,
// 128 codes = four scale blocks, one 16-byte block per lane; a 4x4 word
// transpose inside the quad (three shuffles) then gives lane c bytes 4c..4c+3
// of each block (codes 8c..8c+7), so the 16 k-slots of one MMA all come from
// one block.
// cvt.rn.f16x2.e2m1x2 widens a byte to two fp16 values (low nibble -> low
// half), exactly: the E2M1 magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  A
// block's two MMAs start from zero, and its scale 2^(s-127) multiplies their
// fp32 sum: the products are exact and only fp32 sums round, for every E8M0
// exponent 0..254.
//
// Activations.  Each token row fed to the tensor cores (x for gate/up, h for
// down) is staged in shared memory as fp16 after multiplying it by a power of
// two chosen from the row's largest magnitude (which lands in [1, 2)); the
// fp32 accumulators of that token are multiplied by the inverse power.  bf16
// elements down to 2^-17 of their row's largest pass through unchanged,
// smaller ones round at 2^-25 of it, and h keeps 11 significant bits.
//
// MMA (m16n8k16, fp16 operands, fp32 accumulate; A = weights, B = tokens):
//   gate/up: A rows 0-7 = 8 gate rows of d_ff, rows 8-15 = the same 8 up rows,
//            so the lane holding g also holds u and forms h = silu(g) * u.
//   down:    A rows = 16 consecutive rows of d.
// Lane c's byte b of block q feeds the block's MMA b >> 1, k-slots {2c, 2c+1}
// when b is even and {2c+8, 2c+9} when odd.  The token rows in shared memory
// are read with the same k permutation: one 16-byte load (elements
// 32q + 8c .. +8 of the chunk) per block and token tile.
//
// Units.  gate/up: (woken expert, 8 * 4/ks rows of d_ff); the CTA's 4 warps are
// (4/ks row groups) x (ks parts of d), ks in {1, 2, 4} chosen by the host so
// that small blocks still spread over the GPU; partial sums of the ks parts
// are added in fixed order in shared memory.  down: (woken expert, 64 rows of
// d), one warp per 16 rows over the whole d_ff, the same per-tile ticket and
// slot-ordered combine as the bf16 kernels.
#include "ffn_common.cuh"
#include "mxfp4_common.cuh"

namespace dfv {
namespace {

constexpr int kMxThreads = 128;
constexpr int kMxWarps = 4;
constexpr int kMxBatch = 8;  // 128-code chunks in flight per lane and row

// Streaming 16-byte load, not kept in L1 (every weight byte is used once).
__device__ __forceinline__ uint4 ldg16(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// 4x4 word transpose inside a quad: lane c enters with the four words of block
// c and leaves with word c of blocks 0..3.  Rotate the own words left by c;
// the i-th shuffle (i = 1..3) takes word i from lane (c - i) & 3, which is
// word c of block (c - i) & 3; a rotation right by c of the reversed list then
// orders them by block.
__device__ __forceinline__ uint4 quad_transpose(uint4 w, int c, int lane) {
  const bool r1 = c & 1, r2 = c & 2;
  uint32_t a0 = r1 ? w.y : w.x, a1 = r1 ? w.z : w.y, a2 = r1 ? w.w : w.z, a3 = r1 ? w.x : w.w;
  const uint32_t q0 = r2 ? a2 : a0, q1 = r2 ? a3 : a1, q2 = r2 ? a0 : a2, q3 = r2 ? a1 : a3;
  const int base = lane & ~3;
  const uint32_t v1 = __shfl_sync(0xffffffffu, q1, base | ((c - 1) & 3));
  const uint32_t v2 = __shfl_sync(0xffffffffu, q2, base | ((c - 2) & 3));
  const uint32_t v3 = __shfl_sync(0xffffffffu, q3, base | ((c - 3) & 3));
  // reversed: u[j] = v[(-j) & 3] = {q0, v3, v2, v1}; block q is u[(q - c) & 3]
  a0 = r1 ? v1 : q0;  // rotate right by 1 when c is odd: {v1, q0, v3, v2}
  a1 = r1 ? q0 : v3;
  a2 = r1 ? v3 : v2;
  a3 = r1 ? v2 : v1;
  return r2 ? make_uint4(a2, a3, a0, a1) : make_uint4(a0, a1, a2, a3);
}

// E8M0 byte s -> 2^(s-127) in fp32 (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_f32(uint32_t s) { return __uint_as_float(max(s << 23, 0x00400000u)); }

// 16-byte chunk q of staged token row j: odd rows are offset by four chunks,
// so a quarter-warp (rows j, j+1, lanes c = 0..3 reading chunks 4q'..4q'+3)
// covers all 32 banks.
__device__ __forceinline__ int swz_mx(int q, int j) { return q ^ ((j & 1) << 2); }

// D = A * B (fp16, fp32 accumulate) from zero.
__device__ __forceinline__ void mma_f16_0(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// One block of a lane: acc[0..1] += fa * (A_lo . B), acc[2..3] += fb * (A_hi . B)
// over the block's two MMAs, which start from zero.
__device__ __forceinline__ void mx_block(float (&acc)[4], const uint32_t (&ra)[4], const uint32_t (&rb)[4],
                                         const uint4 &bx, float fa, float fb) {
  float t1[4], t2[4];
  mma_f16_0(t1, ra[0], rb[0], ra[1], rb[1], bx.x, bx.y);
  mma_f16_0(t2, ra[2], rb[2], ra[3], rb[3], bx.z, bx.w);
  acc[0] = fmaf(fa, t1[0] + t2[0], acc[0]);
  acc[1] = fmaf(fa, t1[1] + t2[1], acc[1]);
  acc[2] = fmaf(fb, t1[2] + t2[2], acc[2]);
  acc[3] = fmaf(fb, t1[3] + t2[3], acc[3]);
}

// ----------------------------------------------------------------------------
// gate/up.  Dynamic smem: xs[NT*8][d] fp16 (swizzled) | red[4][NT][32][4] fp32.
template <int NT>
__global__ void __launch_bounds__(kMxThreads) gateup_mxfp4_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = p.d, I = p.I, K = p.K, ks = p.ks;
  const int cpr = d / 8;  // 16-byte fp16 chunks per staged row
  uint4 *xs = reinterpret_cast<uint4 *>(smem);
  float *red = reinterpret_cast<float *>(smem + (size_t)NT * 8 * d * 2);
  __shared__ int s_tok[NT * 8];
  __shared__ float s_inv[NT * 8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int rg = warp / ks, kp = warp - rg * ks;
  const int R = 8 * (kMxWarps / ks);  // d_ff rows per unit
  const int tiles = I / R;
  const int nW = *p.ws.n_woken;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const int C = (d + 127) / 128;  // 128-code chunks per row
  const int c0 = kp * C / ks, c1 = (kp + 1) * C / ks;
  const size_t rowb = (size_t)d / 2;  // code bytes per row
  const int srow = d / 32;            // scale bytes per row
  const uint16_t *xg = reinterpret_cast<const uint16_t *>(p.x);

  int cur = -1, m = 0, off = 0, e = 0;
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, tile = u - wi * tiles;
    if (wi != cur) {
      __syncthreads();
      cur = wi;
      e = p.ws.woken[wi];
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      if (tid < m) s_tok[tid] = pair_token(p.ws.gather[off + tid], p.k, K);
      __syncthreads();
      for (int j = warp; j < m; j += kMxWarps) {
        const uint16_t *src = xg + (size_t)s_tok[j] * d;
        float amax = 0.f;
        for (int q = lane; q < cpr; q += 32) {
          const uint4 v = *reinterpret_cast<const uint4 *>(src + q * 8);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        }
        const int sh = row_shift(warp_max(amax));
        const float sc = exp2i(sh);
        for (int q = lane; q < cpr; q += 32) {
          const uint4 v = *reinterpret_cast<const uint4 *>(src + q * 8);
          xs[j * cpr + swz_mx(q, j)] = make_uint4(pack_h2(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc),
                                               pack_h2(bf16_lo(v.y) * sc, bf16_hi(v.y) * sc),
                                               pack_h2(bf16_lo(v.z) * sc, bf16_hi(v.z) * sc),
                                               pack_h2(bf16_lo(v.w) * sc, bf16_hi(v.w) * sc));
        }
        if (lane == 0) s_inv[j] = exp2i(-sh);
      }
      __syncthreads();
    }
    const int i0 = tile * R + rg * 8;
    const size_t row = (size_t)e * I + i0 + g;
    const uint8_t *pg = reinterpret_cast<const uint8_t *>(p.wg) + row * rowb + c * 16;
    const uint8_t *pu = reinterpret_cast<const uint8_t *>(p.wu) + row * rowb + c * 16;
    const uint8_t *sgp = p.sg + row * srow + c;
    const uint8_t *sup = p.su + row * srow + c;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    for (int base = c0; base < c1; base += kMxBatch) {
      uint4 ag[kMxBatch], au[kMxBatch];
      uint32_t eg[kMxBatch], eu[kMxBatch];
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        ag[j] = au[j] = make_uint4(0u, 0u, 0u, 0u);
        eg[j] = eu[j] = 127u;
        if (ch < c1) {
          // lane c: word c of each block q of the chunk (a block is live when
          // it starts inside the row), and the scale of block c
          const int nb = min(4, (d - ch * 128) / 32);
          if (c < nb) {
            ag[j] = ldg16(pg + (size_t)ch * 64);
            au[j] = ldg16(pu + (size_t)ch * 64);
            eg[j] = ldg_scale(sgp + ch * 4);
            eu[j] = ldg_scale(sup + ch * 4);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        if (ch < c1) {
          const int nb = min(4, (d - ch * 128) / 32);  // live blocks of the chunk (quad-uniform)
          const uint4 tg = quad_transpose(ag[j], c, lane), tu = quad_transpose(au[j], c, lane);
          const uint32_t wg4[4] = {tg.x, tg.y, tg.z, tg.w};
          const uint32_t wu4[4] = {tu.x, tu.y, tu.z, tu.w};
#pragma unroll
          for (int qb = 0; qb < 4; ++qb) {
            // block qb's scales sit with lane qb of the quad
            const float fg = e8m0_f32(__shfl_sync(0xffffffffu, eg[j], (lane & ~3) | qb));
            const float fu = e8m0_f32(__shfl_sync(0xffffffffu, eu[j], (lane & ~3) | qb));
            if (qb < nb) {
              uint32_t rg4[4], ru4[4];
              e2m1_word(wg4[qb], rg4);
              e2m1_word(wu4[qb], ru4);
              const int q = ch * 16 + qb * 4 + c;  // x chunk: elements 128ch + 32qb + 8c .. +8
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt * 8 < m) {
                  const int n = nt * 8 + g;
                  uint4 bx = make_uint4(0u, 0u, 0u, 0u);
                  if (n < m) bx = xs[n * cpr + swz_mx(q, n)];
                  mx_block(acc[nt], rg4, ru4, bx, fg, fu);
                }
              }
            }
          }
        }
      }
    }

    if (ks == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = nt * 8 + 2 * c + q;
          if (tok < m) {
            const float inv = s_inv[tok];
            p.ws.h[(size_t)(off + tok) * I + i0 + g] = silu(acc[nt][q] * inv) * (acc[nt][q + 2] * inv);
          }
        }
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4 *>(red + ((warp * NT + nt) * 32 + lane) * 4) =
            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      __syncthreads();
      const int ngrp = kMxWarps / ks;
      for (int idx = tid; idx < ngrp * NT * 64; idx += kMxThreads) {
        const int r = idx / (NT * 64), rem = idx - r * NT * 64;
        const int nt = rem >> 6, ln = (rem >> 1) & 31, q = rem & 1;
        const int tok = nt * 8 + 2 * (ln & 3) + q;
        if (tok < m) {
          float gs = 0.f, us = 0.f;
          for (int kk = 0; kk < ks; ++kk) {
            const float *rr = red + (((r * ks + kk) * NT + nt) * 32 + ln) * 4;
            gs += rr[q];
            us += rr[q + 2];
          }
          const float inv = s_inv[tok];
          p.ws.h[(size_t)(off + tok) * I + tile * R + r * 8 + (ln >> 2)] = silu(gs * inv) * (us * inv);
        }
      }
      __syncthreads();
    }
  }
}

// ----------------------------------------------------------------------------
// down + combine.  Dynamic smem: hs[NT*8][d_ff] fp16 (swizzled).
template <int NT>
__global__ void __launch_bounds__(kMxThreads, 1) down_mxfp4_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = p.d, I = p.I;
  const int cpr = I / 8;
  uint4 *hs = reinterpret_cast<uint4 *>(smem);
  __shared__ float s_inv[NT * 8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nW = *p.ws.n_woken;
  const int tiles = d / kDownTile;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const int C = (I + 127) / 128;
  const size_t rowb = (size_t)I / 2;
  const int srow = I / 32;

  int cur = -1, m = 0, off = 0, e = 0;
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, dt = u - wi * tiles;
    if (wi != cur) {
      __syncthreads();
      cur = wi;
      e = p.ws.woken[wi];
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      for (int j = warp; j < m; j += kMxWarps) {
        const float *src = p.ws.h + (size_t)(off + j) * I;
        float amax = 0.f;
        for (int q = lane; q < cpr; q += 32) {
          const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8));
          const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8 + 4));
          amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                                   fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w)))));
        }
        const int sh = row_shift(warp_max(amax));
        const float sc = exp2i(sh);
        for (int q = lane; q < cpr; q += 32) {
          const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8));
          const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(src + q * 8 + 4));
          hs[j * cpr + swz_mx(q, j)] = make_uint4(pack_h2(v0.x * sc, v0.y * sc), pack_h2(v0.z * sc, v0.w * sc),
                                               pack_h2(v1.x * sc, v1.y * sc), pack_h2(v1.z * sc, v1.w * sc));
        }
        if (lane == 0) s_inv[j] = exp2i(-sh);
      }
      __syncthreads();
    }
    const int r0 = dt * kDownTile + warp * 16;
    const size_t row = (size_t)e * d + r0 + g;
    const uint8_t *pa = reinterpret_cast<const uint8_t *>(p.wd) + row * rowb + c * 16;
    const uint8_t *pb = pa + 8 * rowb;
    const uint8_t *sap = p.sd + row * srow + c;
    const uint8_t *sbp = sap + 8 * srow;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    for (int base = 0; base < C; base += kMxBatch) {
      uint4 a0[kMxBatch], a1[kMxBatch];
      uint32_t e0[kMxBatch], e1[kMxBatch];
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        a0[j] = a1[j] = make_uint4(0u, 0u, 0u, 0u);
        e0[j] = e1[j] = 127u;
        if (ch < C) {
          const int nb = min(4, (I - ch * 128) / 32);
          if (c < nb) {
            a0[j] = ldg16(pa + (size_t)ch * 64);
            a1[j] = ldg16(pb + (size_t)ch * 64);
            e0[j] = ldg_scale(sap + ch * 4);
            e1[j] = ldg_scale(sbp + ch * 4);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        if (ch < C) {
          const int nb = min(4, (I - ch * 128) / 32);
          const uint4 t0 = quad_transpose(a0[j], c, lane), t1 = quad_transpose(a1[j], c, lane);
          const uint32_t w0[4] = {t0.x, t0.y, t0.z, t0.w};
          const uint32_t w1[4] = {t1.x, t1.y, t1.z, t1.w};
#pragma unroll
          for (int qb = 0; qb < 4; ++qb) {
            const float f0 = e8m0_f32(__shfl_sync(0xffffffffu, e0[j], (lane & ~3) | qb));
            const float f1 = e8m0_f32(__shfl_sync(0xffffffffu, e1[j], (lane & ~3) | qb));
            if (qb < nb) {
              uint32_t r0v[4], r1v[4];
              e2m1_word(w0[qb], r0v);
              e2m1_word(w1[qb], r1v);
              const int q = ch * 16 + qb * 4 + c;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt * 8 < m) {
                  const int n = nt * 8 + g;
                  uint4 bh = make_uint4(0u, 0u, 0u, 0u);
                  if (n < m) bh = hs[n * cpr + swz_mx(q, n)];
                  mx_block(acc[nt], r0v, r1v, bh, f0, f1);
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int tok = nt * 8 + 2 * c + q;
        if (tok < m) {
          const int pair = p.ws.gather[off + tok];
          const float w = p.ws.topk_w[pair] * s_inv[tok];
          p.ws.ys[(size_t)pair * d + r0 + g] = w * acc[nt][q];
          p.ws.ys[(size_t)pair * d + r0 + g + 8] = w * acc[nt][q + 2];
        }
      }
    finish_down_unit(p, dt, nW);
  }
}

size_t mx_gate_smem(int nt, int d) { return (size_t)nt * 8 * d * 2 + (size_t)kMxWarps * nt * 32 * 16; }
size_t mx_down_smem(int nt, int I) { return (size_t)nt * 8 * I * 2; }

}  // namespace

int mxfp4_threads() { return kMxThreads; }

int mxfp4_grid_limit(int k, int d, int I, int which) {
  if (which == 0)
    return k <= 8 ? occupancy_grid(gateup_mxfp4_kernel<1>, kMxThreads, mx_gate_smem(1, d))
                  : occupancy_grid(gateup_mxfp4_kernel<2>, kMxThreads, mx_gate_smem(2, d));
  return k <= 8 ? occupancy_grid(down_mxfp4_kernel<1>, kMxThreads, mx_down_smem(1, I))
                : occupancy_grid(down_mxfp4_kernel<2>, kMxThreads, mx_down_smem(2, I));
}

cudaError_t launch_ffn_mxfp4(const FfnParams &p, int phase, int grid, cudaStream_t s, bool pdl) {
  cudaError_t err;
  const bool one = p.k <= 8;
  if (phase == 0) {
    if (p.ks != 1 && p.ks != 2 && p.ks != 4) return cudaErrorInvalidValue;
    const size_t sm = mx_gate_smem(one ? 1 : 2, p.d);
    if (one) {
      if ((err = ensure_smem(gateup_mxfp4_kernel<1>, sm)) != cudaSuccess) return err;
      return launch_ffn_kernel(gateup_mxfp4_kernel<1>, grid, kMxThreads, sm, p, s, pdl);
    }
    if ((err = ensure_smem(gateup_mxfp4_kernel<2>, sm)) != cudaSuccess) return err;
    return launch_ffn_kernel(gateup_mxfp4_kernel<2>, grid, kMxThreads, sm, p, s, pdl);
  }
  const size_t sm = mx_down_smem(one ? 1 : 2, p.I);
  if (one) {
    if ((err = ensure_smem(down_mxfp4_kernel<1>, sm)) != cudaSuccess) return err;
    return launch_ffn_kernel(down_mxfp4_kernel<1>, grid, kMxThreads, sm, p, s, pdl);
  }
  if ((err = ensure_smem(down_mxfp4_kernel<2>, sm)) != cudaSuccess) return err;
  return launch_ffn_kernel(down_mxfp4_kernel<2>, grid, kMxThreads, sm, p, s, pdl);
}

}  // namespace dfv
