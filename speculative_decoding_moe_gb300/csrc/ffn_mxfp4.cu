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
// Decode.  One 16-byte load of a lane holds 32 codes of one row, i.e. exactly
// one scale block.  cvt.rn.f16x2.e2m1x2 widens a byte to two fp16 values
// (low nibble -> low half), exactly: the E2M1 magnitudes are
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  One fp16x2 multiply by the block's scale
// 2^(s-127) keeps them exact as long as the scale is a normal fp16 number and
// every product a normal one or a subnormal on the 2^-24 grid, which holds for
// s in [113, 140].  A scale outside that range sets DFV_DEVERR_SCALE_RANGE in
// the workspace error word (the outputs are then wrong).
//
// Activations.  Each token row fed to the tensor cores (x for gate/up, h for
// down) is staged in shared memory as fp16 after multiplying it by a power of
// two chosen from the row's largest magnitude (which lands in [2^14, 2^15));
// the fp32 accumulators of that token are multiplied by the inverse power.
// Both scalings are exact, so the bf16 rows x pass through unchanged and h
// keeps 11 significant bits.
//
// MMA (m16n8k16, fp16 operands, fp32 accumulate; A = weights, B = tokens):
//   gate/up: A rows 0-7 = 8 gate rows of d_ff, rows 8-15 = the same 8 up rows,
//            so the lane holding g also holds u and forms h = silu(g) * u.
//   down:    A rows = 16 consecutive rows of d.
// The four lanes c = 0..3 of a quad read 64 contiguous bytes (128 codes) of a
// row; lane c holds codes [32c, 32c + 32).  Its byte 4t + b (t = 0..3) feeds
// MMA 2t + (b >> 1), k-slots {2c, 2c+1} when b is even and {2c+8, 2c+9} when
// odd.  The token rows in shared memory are read with the same k permutation:
// one 16-byte load (codes 32c + 8t .. +8) per two MMAs.
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
  uint32_t range = 0;

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
          xs[j * cpr + swz(q, j)] = make_uint4(pack_h2(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc),
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
        if (ch < c1 && ch * 128 + c * 32 < d) {
          ag[j] = ldg_codes(pg + (size_t)ch * 64);
          au[j] = ldg_codes(pu + (size_t)ch * 64);
          eg[j] = ldg_scale(sgp + ch * 4);
          eu[j] = ldg_scale(sup + ch * 4);
        }
      }
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        if (ch < c1) {
          const bool live = ch * 128 + c * 32 < d;
          const uint32_t sgv = e8m0_half2(eg[j], range), suv = e8m0_half2(eu[j], range);
          const uint32_t wg4[4] = {ag[j].x, ag[j].y, ag[j].z, ag[j].w};
          const uint32_t wu4[4] = {au[j].x, au[j].y, au[j].z, au[j].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t rg4[4], ru4[4];
            e2m1_word(wg4[t], rg4);
            e2m1_word(wu4[t], ru4);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              rg4[b] = hmul2(rg4[b], sgv);
              ru4[b] = hmul2(ru4[b], suv);
            }
            const int q = ch * 16 + c * 4 + t;  // x chunk: codes 128ch + 32c + 8t .. +8
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (nt * 8 < m) {
                const int n = nt * 8 + g;
                uint4 bx = make_uint4(0u, 0u, 0u, 0u);
                if (n < m && live) bx = xs[n * cpr + swz(q, n)];
                mma_f16x(acc[nt], rg4[0], ru4[0], rg4[1], ru4[1], bx.x, bx.y);
                mma_f16x(acc[nt], rg4[2], ru4[2], rg4[3], ru4[3], bx.z, bx.w);
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
  if (range > kScaleRangeMax) atomicOr(p.ws.err, DFV_DEVERR_SCALE_RANGE);
}

// ----------------------------------------------------------------------------
// down + combine.  Dynamic smem: hs[NT*8][d_ff] fp16 (swizzled).
template <int NT>
__global__ void __launch_bounds__(kMxThreads) down_mxfp4_kernel(FfnParams p) {
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
  uint32_t range = 0;

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
          hs[j * cpr + swz(q, j)] = make_uint4(pack_h2(v0.x * sc, v0.y * sc), pack_h2(v0.z * sc, v0.w * sc),
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
        if (ch < C && ch * 128 + c * 32 < I) {
          a0[j] = ldg_codes(pa + (size_t)ch * 64);
          a1[j] = ldg_codes(pb + (size_t)ch * 64);
          e0[j] = ldg_scale(sap + ch * 4);
          e1[j] = ldg_scale(sbp + ch * 4);
        }
      }
#pragma unroll
      for (int j = 0; j < kMxBatch; ++j) {
        const int ch = base + j;
        if (ch < C) {
          const bool live = ch * 128 + c * 32 < I;
          const uint32_t s0 = e8m0_half2(e0[j], range), s1 = e8m0_half2(e1[j], range);
          const uint32_t w0[4] = {a0[j].x, a0[j].y, a0[j].z, a0[j].w};
          const uint32_t w1[4] = {a1[j].x, a1[j].y, a1[j].z, a1[j].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t r0v[4], r1v[4];
            e2m1_word(w0[t], r0v);
            e2m1_word(w1[t], r1v);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              r0v[b] = hmul2(r0v[b], s0);
              r1v[b] = hmul2(r1v[b], s1);
            }
            const int q = ch * 16 + c * 4 + t;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (nt * 8 < m) {
                const int n = nt * 8 + g;
                uint4 bh = make_uint4(0u, 0u, 0u, 0u);
                if (n < m && live) bh = hs[n * cpr + swz(q, n)];
                mma_f16x(acc[nt], r0v[0], r1v[0], r0v[1], r1v[1], bh.x, bh.y);
                mma_f16x(acc[nt], r0v[2], r1v[2], r0v[3], r1v[3], bh.z, bh.w);
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
  if (range > kScaleRangeMax) atomicOr(p.ws.err, DFV_DEVERR_SCALE_RANGE);
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
