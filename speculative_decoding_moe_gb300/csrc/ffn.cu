// ffn.cu -- grouped SwiGLU expert FFN and routing-weighted combine over the
// woken experts of a verify block.
//
// "Speculating on a Strix Halo", section "The verify's own cost": the tokens
// of the block are sorted by expert and each projection runs as one grouped
// launch; section "What the pieces cost": the block wakes the union of its
// rows' experts and each token's output is the routing-weighted sum of its K
// experts.  Part 2, section "The verification cog": the cost is streaming the
// woken experts' weights, so every weight byte is read from HBM exactly once.
//
// Two launches per layer (chained with programmatic dependent launch):
//   gate/up:  unit = (woken expert, 8 d_ff rows).  One m16n8k16 tile holds the
//             8 gate rows (M rows 0-7) and the 8 up rows (M rows 8-15), so
//             h = silu(g) * u is formed in the thread that owns both.  The
//             tokens of the expert are the N columns (<= 8 per tile, zero
//             padded); d is split over the CTA's 8 warps and the warp partials
//             are summed in fixed order in shared memory.
//   down:     unit = (woken expert, 64 d rows); 4 row-warps x 2 k-halves.  h is
//             staged as a bf16 hi/lo pair so the down product keeps ~16 bits
//             of h.  The weighted result of each (token, slot) pair goes to
//             ys[pair][row]; the last unit to finish a 64-row tile (atomic
//             ticket, no waiting) sums ys over the K slots in slot order and
//             writes out (plus an optional residual).
//
// Weights are read straight from HBM into the MMA A fragments with 128-bit
// non-coherent loads, no L1 allocation, eight 32-element k-chunks in flight per
// thread.  The k index inside a 32-element chunk is permuted identically on the
// A (weights) and B (tokens) side, so each thread's 16-byte load feeds two
// MMAs without any shuffle.
#include "ffn_common.cuh"

namespace dfv {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kBatch = 8;  // 32-element k-chunks per load batch

// ----------------------------------------------------------------------------
// bf16 gate/up.  Dynamic smem: xs[NT*8][d] bf16 (16-byte chunks XOR-swizzled
// by row parity when d % 64 == 0) | red[8][NT][32][4] fp32.
template <int NT>
__global__ void __launch_bounds__(kThreads) gateup_bf16_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = p.d, I = p.I, K = p.K;
  const int cpr = d / 8;  // 16-byte chunks per x row
  uint4 *xs = reinterpret_cast<uint4 *>(smem);
  float *red = reinterpret_cast<float *>(smem + (size_t)NT * 8 * d * 2);
  __shared__ int s_tok[NT * 8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nW = *p.ws.n_woken;
  const int tiles = I / kGateTile;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const int C = d / 32;
  const int c0 = warp * C / kWarps, c1 = (warp + 1) * C / kWarps;
  const uint16_t *xg = reinterpret_cast<const uint16_t *>(p.x);

  int cur = -1, m = 0, off = 0, e = 0;
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, tile = u % tiles;
    if (wi != cur) {
      __syncthreads();
      cur = wi;
      e = p.ws.woken[wi];
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      if (tid < m) s_tok[tid] = pair_token(p.ws.gather[off + tid], p.k, K);
      __syncthreads();
      for (int idx = tid; idx < m * cpr; idx += kThreads) {
        const int j = idx / cpr, q = idx % cpr;
        const uint4 v = *reinterpret_cast<const uint4 *>(xg + (size_t)s_tok[j] * d + q * 8);
        xs[j * cpr + (q ^ ((j & 1) ? p.swz_x : 0))] = v;
      }
      __syncthreads();
    }
    const int i0 = tile * kGateTile;
    const uint16_t *pg = reinterpret_cast<const uint16_t *>(p.wg) + ((size_t)e * I + i0 + g) * d + c * 8;
    const uint16_t *pu = reinterpret_cast<const uint16_t *>(p.wu) + ((size_t)e * I + i0 + g) * d + c * 8;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    for (int base = c0; base < c1; base += kBatch) {
      uint4 ag[kBatch], au[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (base + j < c1) {
          ag[j] = ldg_stream(pg + (size_t)(base + j) * 32);
          au[j] = ldg_stream(pu + (size_t)(base + j) * 32);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (base + j < c1) {
          const int q = (base + j) * 4 + c;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt * 8 < m) {
              const int row = nt * 8 + g;
              uint4 b = make_uint4(0u, 0u, 0u, 0u);
              if (row < m) b = xs[row * cpr + (q ^ ((row & 1) ? p.swz_x : 0))];
              mma_bf16(acc[nt], ag[j].x, au[j].x, ag[j].y, au[j].y, b.x, b.y);
              mma_bf16(acc[nt], ag[j].z, au[j].z, ag[j].w, au[j].w, b.z, b.w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4 *>(red + ((warp * NT + nt) * 32 + lane) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    __syncthreads();
    if (tid < NT * 64) {
      const int nt = tid >> 6, ln = (tid >> 1) & 31, q = tid & 1;
      const int tok = nt * 8 + 2 * (ln & 3) + q;
      if (tok < m) {
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          gs += red[((w * NT + nt) * 32 + ln) * 4 + q];
          us += red[((w * NT + nt) * 32 + ln) * 4 + q + 2];
        }
        p.ws.h[(size_t)(off + tok) * I + i0 + (ln >> 2)] = silu(gs) * us;
      }
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------
// bf16 down + combine.  Dynamic smem: hh[NT*8][I] bf16 | hl[NT*8][I] bf16 |
// red[2][4][NT][32][4] fp32.
template <int NT>
__global__ void __launch_bounds__(kThreads) down_bf16_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = p.d, I = p.I;
  const int cpr = I / 8;
  uint4 *hh = reinterpret_cast<uint4 *>(smem);
  uint4 *hl = reinterpret_cast<uint4 *>(smem + (size_t)NT * 8 * I * 2);
  float *red = reinterpret_cast<float *>(smem + (size_t)NT * 8 * I * 4);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int rw = warp & 3, kw = warp >> 2;
  const int nW = *p.ws.n_woken;
  const int tiles = (d + kDownTile - 1) / kDownTile;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const int C = I / 32;
  const int c0 = kw * C / 2, c1 = (kw + 1) * C / 2;

  int cur = -1, m = 0, off = 0, e = 0;
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, dt = u % tiles;
    if (wi != cur) {
      __syncthreads();
      cur = wi;
      e = p.ws.woken[wi];
      off = p.ws.offsets[wi];
      m = p.ws.offsets[wi + 1] - off;
      for (int idx = tid; idx < m * cpr; idx += kThreads) {
        const int j = idx / cpr, q = idx % cpr;
        const float4 *src = reinterpret_cast<const float4 *>(p.ws.h + (size_t)(off + j) * I + q * 8);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t h2[4], l2[4];
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const __nv_bfloat16 a = __float2bfloat16_rn(v[2 * q2]), b = __float2bfloat16_rn(v[2 * q2 + 1]);
          const __nv_bfloat16 la = __float2bfloat16_rn(v[2 * q2] - __bfloat162float(a));
          const __nv_bfloat16 lb = __float2bfloat16_rn(v[2 * q2 + 1] - __bfloat162float(b));
          h2[q2] = (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
          l2[q2] = (uint32_t)__bfloat16_as_ushort(la) | ((uint32_t)__bfloat16_as_ushort(lb) << 16);
        }
        const int qq = q ^ ((j & 1) ? p.swz_h : 0);
        hh[j * cpr + qq] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
        hl[j * cpr + qq] = make_uint4(l2[0], l2[1], l2[2], l2[3]);
      }
      __syncthreads();
    }
    const int r0 = dt * kDownTile + rw * 16;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    if (r0 < d) {
      const uint16_t *pa = reinterpret_cast<const uint16_t *>(p.wd) + ((size_t)e * d + r0 + g) * I + c * 8;
      const uint16_t *pb = pa + (size_t)8 * I;
      for (int base = c0; base < c1; base += kBatch) {
        uint4 a0[kBatch], a1[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          if (base + j < c1) {
            a0[j] = ldg_stream(pa + (size_t)(base + j) * 32);
            a1[j] = ldg_stream(pb + (size_t)(base + j) * 32);
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          if (base + j < c1) {
            const int q = (base + j) * 4 + c;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (nt * 8 < m) {
                const int row = nt * 8 + g;
                uint4 bh = make_uint4(0u, 0u, 0u, 0u), bl = bh;
                if (row < m) {
                  const int qq = row * cpr + (q ^ ((row & 1) ? p.swz_h : 0));
                  bh = hh[qq];
                  bl = hl[qq];
                }
                mma_bf16(acc[nt], a0[j].x, a1[j].x, a0[j].y, a1[j].y, bh.x, bh.y);
                mma_bf16(acc[nt], a0[j].z, a1[j].z, a0[j].w, a1[j].w, bh.z, bh.w);
                mma_bf16(acc[nt], a0[j].x, a1[j].x, a0[j].y, a1[j].y, bl.x, bl.y);
                mma_bf16(acc[nt], a0[j].z, a1[j].z, a0[j].w, a1[j].w, bl.z, bl.w);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4 *>(red + (((kw * 4 + rw) * NT + nt) * 32 + lane) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    __syncthreads();
    for (int idx = tid; idx < 4 * NT * 32 * 4; idx += kThreads) {
      const int q4 = idx & 3, ln = (idx >> 2) & 31, nt = (idx >> 7) % NT, rws = idx / (128 * NT);
      const int row = dt * kDownTile + rws * 16 + (ln >> 2) + ((q4 & 2) ? 8 : 0);
      const int tok = nt * 8 + 2 * (ln & 3) + (q4 & 1);
      if (tok < m && row < d) {
        const float y = red[(((0 * 4 + rws) * NT + nt) * 32 + ln) * 4 + q4] +
                        red[(((1 * 4 + rws) * NT + nt) * 32 + ln) * 4 + q4];
        const int pair = p.ws.gather[off + tok];
        p.ws.ys[(size_t)pair * d + row] = p.ws.topk_w[pair] * y;
      }
    }
    finish_down_unit(p, dt, nW);
  }
}

// ----------------------------------------------------------------------------
// fp32 weights: plain CUDA-core kernels (small layers; not the bandwidth path).
__global__ void __launch_bounds__(kThreads) gateup_f32_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  const int d = p.d, I = p.I, K = p.K;
  const int nW = *p.ws.n_woken;
  const int tiles = I / kGateTile;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const float *x = reinterpret_cast<const float *>(p.x);
  const float *wg = reinterpret_cast<const float *>(p.wg);
  const float *wu = reinterpret_cast<const float *>(p.wu);
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, i0 = (u % tiles) * kGateTile;
    const int e = p.ws.woken[wi], off = p.ws.offsets[wi], m = p.ws.offsets[wi + 1] - off;
    const int rho = threadIdx.x >> 4, j = threadIdx.x & 15;  // 16 rows x 16 tokens
    if (rho < kGateTile && j < m) {
      const int t = pair_token(p.ws.gather[off + j], p.k, K);
      const float *xr = x + (size_t)t * d;
      const float *gr = wg + ((size_t)e * I + i0 + rho) * d;
      const float *ur = wu + ((size_t)e * I + i0 + rho) * d;
      float gs = 0.f, us = 0.f;
      for (int kk = 0; kk < d; ++kk) {
        gs = fmaf(xr[kk], gr[kk], gs);
        us = fmaf(xr[kk], ur[kk], us);
      }
      p.ws.h[(size_t)(off + j) * I + i0 + rho] = silu(gs) * us;
    }
  }
}

__global__ void __launch_bounds__(kThreads) down_f32_kernel(FfnParams p) {
  pdl_trigger();
  pdl_wait();
  const int d = p.d, I = p.I;
  const int nW = *p.ws.n_woken;
  const int tiles = (d + kDownTile - 1) / kDownTile;
  int lo, hi;
  unit_range(nW * tiles, lo, hi);
  const float *wd = reinterpret_cast<const float *>(p.wd);
  for (int u = lo; u < hi; ++u) {
    const int wi = u / tiles, dt = u % tiles;
    const int e = p.ws.woken[wi], off = p.ws.offsets[wi], m = p.ws.offsets[wi + 1] - off;
    const int rr = threadIdx.x & 63, jg = threadIdx.x >> 6;
    const int r = dt * kDownTile + rr;
    if (r < d) {
      const float *dr = wd + ((size_t)e * d + r) * I;
      for (int j = jg; j < m; j += kThreads / kDownTile) {
        const float *hr = p.ws.h + (size_t)(off + j) * I;
        float y = 0.f;
        for (int i = 0; i < I; ++i) y = fmaf(__ldcg(hr + i), dr[i], y);
        const int pair = p.ws.gather[off + j];
        p.ws.ys[(size_t)pair * d + r] = p.ws.topk_w[pair] * y;
      }
    }
    finish_down_unit(p, dt, nW);
  }
}

// ----------------------------------------------------------------------------
// host side
namespace {

size_t gate_smem(int nt, int d) { return (size_t)nt * 8 * d * 2 + (size_t)kWarps * nt * 32 * 16; }
size_t down_smem(int nt, int I) { return (size_t)nt * 8 * I * 4 + (size_t)8 * nt * 32 * 16; }

template <typename F>
cudaError_t launch(F kern, int grid, size_t smem, const FfnParams &p, cudaStream_t s, bool pdl) {
  return launch_ffn_kernel(kern, grid, kThreads, smem, p, s, pdl);
}

template <typename F>
int occupancy_grid(F kern, size_t smem) {
  return occupancy_grid(kern, kThreads, smem);
}

}  // namespace

int ffn_grid_limit(int w_dtype, int k, int d, int I, int which) {
  const int nt = k <= 8 ? 1 : 2;
  if (w_dtype == DFV_BF16) {
    if (which == 0)
      return nt == 1 ? occupancy_grid(gateup_bf16_kernel<1>, gate_smem(1, d))
                     : occupancy_grid(gateup_bf16_kernel<2>, gate_smem(2, d));
    return nt == 1 ? occupancy_grid(down_bf16_kernel<1>, down_smem(1, I))
                   : occupancy_grid(down_bf16_kernel<2>, down_smem(2, I));
  }
  if (w_dtype == DFV_F32) {
    return which == 0 ? occupancy_grid(gateup_f32_kernel, 0) : occupancy_grid(down_f32_kernel, 0);
  }
  if (w_dtype == DFV_MXFP4) return mxfp4_grid_limit(k, d, I, which);
  return 0;
}

cudaError_t launch_ffn_phase(const FfnParams &p, int w_dtype, int phase, int grid, cudaStream_t s, bool pdl) {
  cudaError_t err;
  if (w_dtype == DFV_BF16) {
    if (p.k <= 8) {
      if (phase == 0) {
        if ((err = ensure_smem(gateup_bf16_kernel<1>, gate_smem(1, p.d))) != cudaSuccess) return err;
        return launch(gateup_bf16_kernel<1>, grid, gate_smem(1, p.d), p, s, pdl);
      }
      if ((err = ensure_smem(down_bf16_kernel<1>, down_smem(1, p.I))) != cudaSuccess) return err;
      return launch(down_bf16_kernel<1>, grid, down_smem(1, p.I), p, s, pdl);
    }
    if (phase == 0) {
      if ((err = ensure_smem(gateup_bf16_kernel<2>, gate_smem(2, p.d))) != cudaSuccess) return err;
      return launch(gateup_bf16_kernel<2>, grid, gate_smem(2, p.d), p, s, pdl);
    }
    if ((err = ensure_smem(down_bf16_kernel<2>, down_smem(2, p.I))) != cudaSuccess) return err;
    return launch(down_bf16_kernel<2>, grid, down_smem(2, p.I), p, s, pdl);
  }
  if (w_dtype == DFV_F32) {
    return phase == 0 ? launch(gateup_f32_kernel, grid, 0, p, s, pdl) : launch(down_f32_kernel, grid, 0, p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dfv
