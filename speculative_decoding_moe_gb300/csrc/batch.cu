// batch.cu -- batched verify: B verify blocks of k positions (T = B * k rows,
// up to 512) through one MoE layer with bf16 experts.  The MI355X / vLLM
// write-up, section "Results: Throughput and Speedup", serves up to 32
// concurrent requests: each woken expert's weights are then streamed once for
// every row of every block that routes to it, and experts see tens of tokens,
// so the expert contractions run on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory) fed by TMA.
//
// Launches, in stream order (chained with programmatic dependent launch):
//   logits   router GEMV of every row, in the same summation order as the
//            single-block kernels (a row's logits, hence its experts, do not
//            depend on the batch), and the per-expert token masks cleared
//   topk     one warp per row: top-K (largest logit, lowest id among equals),
//            renormalised softmax weights, bit t of its experts' token masks
//   tables   one CTA: woken union and pair offsets (block scan), the pair list
//            sorted by (expert, row) from the masks, the shared expert
//            appended, and the work units of the two contractions
//   gather   the x row of every sorted pair, copied to Xg[position]
//   gateup   per unit (woken expert, 128 d_ff rows, <= 128 of its tokens):
//            Dg = Wg_tile . Xg^T and Du = Wu_tile . Xg^T in TMEM (M = 128
//            weight rows, N = the tokens padded to 16, K = d in 64-column
//            stages), H[position][i] = bf16(silu(Dg) * Du)
//   down     per unit (woken expert, 128 d rows, <= 128 tokens):
//            D = Wd_tile . H^T, Ys[pair][r] = w_pair * D
//   combine  out[t] = bf16(sum over slots s of Ys[t*K+s] (+ Ys[T*K+t]))
// Each contraction kernel is persistent (one CTA per SM, units round robin):
// warp 0 streams weight and token tiles with TMA into a ring of stages, one
// thread of warp 1 issues the MMAs and commits each stage back to the
// producer, warps 2-5 read the accumulators out of TMEM; two TMEM buffers let
// the MMAs of one unit run while the epilogue reads the last.  Every wait is
// bounded (2 s) and reports through the workspace error word.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "fused_common.cuh"
#include "tc05.cuh"

namespace dfv {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char *why, size_t why_len);

namespace {

constexpr int kBRowTile = 8;     // router: rows per CTA
constexpr int kBExpTile = 32;    // router: experts per CTA
constexpr int kTcThreads = 192;  // contraction kernels: producer, MMA, 4 epilogue warps
constexpr int kTcK = 64;         // K elements per stage (one 128-byte swizzle row)
constexpr int kTcM = 128;        // weight rows per unit
constexpr int kTcNMax = 128;     // tokens per unit (TMEM: two buffers of one or two accumulators)
constexpr int kTcBoxN = 16;      // token rows per TMA box
constexpr int kTcEpiBar = 1;     // named barrier of the four epilogue warps

// tcgen05 kernels' parameters (tensor maps first: 64-byte aligned in the
// kernel parameter space)
struct TcParams {
  CUtensorMap tm_a1, tm_a2, tm_b;
  const int4 *units;      // (woken index, row tile, first token, tokens)
  const int *n_units;
  const int *woken, *off, *gather;
  const float *w;         // pair weights (down)
  uint16_t *h;            // gate/up output [P][I] bf16
  float *ys;              // down output [P][d] fp32
  unsigned *err;
  int a_rows;             // weight rows per expert (I for gate/up, d for down)
  int kdim;               // contraction length (d for gate/up, I for down)
  int ncols;              // output row length (I for gate/up, d for down)
};

// ---------------------------------------------------------------- router
__global__ void __launch_bounds__(512) batch_logits_kernel(BatchParams p) {
  extern __shared__ __align__(16) unsigned char bsm[];
  pdl_trigger();
  pdl_wait();
  const int T = p.T, d = p.d, E = p.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the token masks the top-K kernel sets are cleared here (stream order)
  {
    const int nmw = (E + 1) * (p.Tmax / 32);
    const int gid = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid, gsz = gridDim.x * gridDim.y * blockDim.x;
    for (int i = gid; i < nmw; i += gsz) p.tmask[i] = 0u;
  }
  const int t0 = blockIdx.x * kBRowTile, nt = min(kBRowTile, T - t0);
  const int e0 = blockIdx.y * kBExpTile, ne = min(kBExpTile, E - e0);
  uint16_t *xs = reinterpret_cast<uint16_t *>(bsm);  // [nt][d]
  const int cpr = d / 8;
  for (int i = tid; i < nt * cpr; i += blockDim.x)
    reinterpret_cast<uint4 *>(xs)[i] = reinterpret_cast<const uint4 *>(p.x)[(size_t)t0 * cpr + i];
  __syncthreads();
  // warp w: experts e0 + w, e0 + w + 16, each dot product in the order the
  // single-block kernels use (lane l: 16-byte pieces l, l+32, ... in chunks
  // of 256 pieces, words in order, then an xor butterfly); a chunk of the
  // router row is loaded once and used for all the tile's rows
  for (int j = warp; j < ne; j += 16) {
    const int e = e0 + j;
    const uint16_t *wr = reinterpret_cast<const uint16_t *>(p.wr) + (size_t)e * d;
    float acc[kBRowTile];
#pragma unroll
    for (int t = 0; t < kBRowTile; ++t) acc[t] = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < cpr; c0 += 256) {
      uint4 wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        wv[i] = c < cpr ? __ldg(reinterpret_cast<const uint4 *>(wr + (size_t)c * 8)) : make_uint4(0u, 0u, 0u, 0u);
      }
      // piece by piece: the piece's router elements are widened once and
      // used for every row of the tile (each row still sums its pieces in
      // order, words in order, low half first)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < cpr) {
          const uint32_t w4[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
          float wf[8];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            wf[2 * h] = bf16_lo(w4[h]);
            wf[2 * h + 1] = bf16_hi(w4[h]);
          }
#pragma unroll
          for (int t = 0; t < kBRowTile; ++t) {
            if (t < nt) {
              const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * d + (size_t)c * 8);
              const uint32_t x4[4] = {xv.x, xv.y, xv.z, xv.w};
              float a_ = acc[t];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                a_ = fmaf(bf16_lo(x4[h]), wf[2 * h], a_);
                a_ = fmaf(bf16_hi(x4[h]), wf[2 * h + 1], a_);
              }
              acc[t] = a_;
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kBRowTile; ++t) {
      float a_ = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a_ += __shfl_xor_sync(0xffffffffu, a_, o);
      if (lane == 0 && t < nt) p.logits[(size_t)(t0 + t) * E + e] = a_;
    }
  }
}

// warp per row: the top-K selection and weights of the single-block kernels
__global__ void __launch_bounds__(512) batch_topk_kernel(BatchParams p) {
  pdl_trigger();
  pdl_wait();
  const int E = p.E, K = p.K, T = p.T;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 16 + (threadIdx.x >> 5);
  if (t >= T) return;
  uint32_t key[8];
  float val[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    val[q] = (e < E) ? p.logits[(size_t)t * E + e] : 0.f;
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
    p.topk_idx[t * K + lane] = sel_id;
    if (p.u_idx) p.u_idx[t * K + lane] = sel_id;
    p.topk_w[t * K + lane] = z / den;
    atomicOr(&p.tmask[(size_t)sel_id * (p.Tmax / 32) + (t >> 5)], 1u << (t & 31));
  }
}

// one CTA of 512 threads: the woken union, offsets, sorted pairs and units
__global__ void __launch_bounds__(512) batch_tables_kernel(BatchParams p) {
  pdl_trigger();
  pdl_wait();
  const int E = p.E, K = p.K, T = p.T, ns = p.ns;
  const int mw = p.Tmax / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int s_cnt[kMaxExperts + 1], s_eoff[kMaxExperts + 1], s_wsum[16], s_csum[16];
  __shared__ int s_nw, s_ug[kMaxExperts + 2], s_ud[kMaxExperts + 2];
  // rows of earlier mask words and the token masks, one padded row per
  // expert (odd word strides: a warp's lookups for different experts spread
  // over the banks)
  __shared__ unsigned short s_pref[kMaxExperts][DFV_MAX_BATCH_ROWS / 32 + 2];
  __shared__ unsigned s_mask[kMaxExperts][DFV_MAX_BATCH_ROWS / 32 + 1];
  int cnt = 0;
  if (tid < E) {
    // all of the expert's mask words in flight at once, then kept in shared memory
    constexpr int kMW = DFV_MAX_BATCH_ROWS / 32;
    const int nw = (T + 31) / 32;
    unsigned mv[kMW];
#pragma unroll
    for (int w = 0; w < kMW; ++w) mv[w] = w < nw ? p.tmask[(size_t)tid * mw + w] : 0u;
#pragma unroll
    for (int w = 0; w < kMW; ++w) {
      s_pref[tid][w] = (unsigned short)cnt;
      s_mask[tid][w] = mv[w];
      cnt += __popc(mv[w]);
    }
  }
  const int flag = cnt > 0;
  int fi = flag, ci = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, fi, o), b = __shfl_up_sync(0xffffffffu, ci, o);
    if (lane >= o) { fi += a; ci += b; }
  }
  if (lane == 31) { s_wsum[warp] = fi; s_csum[warp] = ci; }
  __syncthreads();
  int wb = 0, cb = 0, nW = 0;
  for (int w = 0; w < 16; ++w) {
    if (w < warp) { wb += s_wsum[w]; cb += s_csum[w]; }
    nW += s_wsum[w];
  }
  const int wpos = wb + fi - flag, eoff = cb + ci - cnt;
  if (tid < E) s_eoff[tid] = eoff;
  if (flag) { p.woken[wpos] = tid; p.off[wpos] = eoff; s_cnt[wpos] = cnt; }
  if (tid == 0) {
    int n = nW;
    p.off[n] = T * K;
    if (ns) {  // the shared expert: id E, every row, weight 1, pairs T*K + t
      p.woken[n] = E;
      s_cnt[n] = T;
      ++n;
      p.off[n] = T * K + T;
    }
    s_nw = n;
    *p.n_woken = n;
    if (p.u_nw) *p.u_nw = nW;
  }
  __syncthreads();
  const int nWt = s_nw;
  // sorted pairs: pair t*K+s of expert e lands at eoff[e] + (rows before t
  // that chose e); eight pairs per thread with their expert ids loaded at once
  for (int q0 = 0; q0 < T * K; q0 += 8 * 512) {
    int ev[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = q0 + j * 512 + tid;
      ev[j] = q < T * K ? p.topk_idx[q] : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = q0 + j * 512 + tid;
      if (q < T * K) {
        const int t = q / K, e = ev[j];
        const int rank = s_pref[e][t >> 5] + __popc(s_mask[e][t >> 5] & ((1u << (t & 31)) - 1u));
        p.gather[s_eoff[e] + rank] = q;
      }
    }
  }
  if (ns)
    for (int t = tid; t < T; t += blockDim.x) {
      p.gather[T * K + t] = T * K + t;
      p.topk_w[T * K + t] = 1.f;
    }
  // units: per woken expert, row tiles x passes of <= 128 tokens
  const int tg = p.I / kTcM, td = p.d / kTcM;
  if (warp == 0) {
    // each woken expert's first gate/up and down unit: exclusive scans of its
    // unit counts, 32 experts at a time
    int ug = 0, ud = 0;
    for (int base = 0; base < nWt; base += 32) {
      const int wi = base + lane;
      const int passes = wi < nWt ? (s_cnt[wi] + kTcNMax - 1) / kTcNMax : 0;
      int ig = tg * passes, id = td * passes;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ig, o), b = __shfl_up_sync(0xffffffffu, id, o);
        if (lane >= o) { ig += a; id += b; }
      }
      if (wi < nWt) {
        s_ug[wi] = ug + ig - tg * passes;
        s_ud[wi] = ud + id - td * passes;
      }
      ug += __shfl_sync(0xffffffffu, ig, 31);
      ud += __shfl_sync(0xffffffffu, id, 31);
    }
    if (lane == 0) {
      s_ug[nWt] = ug;
      s_ud[nWt] = ud;
      p.n_units[0] = ug;
      p.n_units[1] = ud;
    }
  }
  __syncthreads();
  // every thread writes units: unit u of a contraction belongs to the woken
  // expert wi with first[wi] <= u < first[wi + 1] (binary search)
  auto write_units = [&](const int *first, int per, int4 *units) {
    const int total = first[nWt];
    for (int u = tid; u < total; u += blockDim.x) {
      int lo = 0, hi = nWt;  // first[lo] <= u < first[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (first[mid] <= u) lo = mid; else hi = mid;
      }
      const int wi = lo, i = u - first[wi], m = s_cnt[wi];
      const int ps = i / per, mt = i - ps * per;
      units[u] = make_int4(wi, mt, ps * kTcNMax, min(kTcNMax, m - ps * kTcNMax));
    }
  };
  write_units(s_ug, tg, p.units_g);
  write_units(s_ud, td, p.units_d);
}

// Xg[position] = x[row of the pair at that position]
__global__ void __launch_bounds__(256) batch_gather_kernel(BatchParams p) {
  pdl_trigger();
  pdl_wait();
  const int P = p.T * p.K + p.ns * p.T, cpr = p.d / 8;
  for (int pos = blockIdx.x; pos < P; pos += gridDim.x) {
    const int q = p.gather[pos];
    const int t = q < p.T * p.K ? q / p.K : q - p.T * p.K;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.x) + (size_t)t * cpr;
    uint4 *dst = reinterpret_cast<uint4 *>(p.xg) + (size_t)pos * cpr;
    for (int c = threadIdx.x; c < cpr; c += blockDim.x) dst[c] = src[c];
  }
}

// out[t][r] = bf16(sum_s ys[t*K+s][r] (+ ys[T*K+t][r]))
__global__ void __launch_bounds__(256) batch_combine_kernel(BatchParams p) {
  pdl_trigger();
  pdl_wait();
  const int T = p.T, K = p.K, d = p.d;
  // four consecutive outputs per thread (d % 128 == 0), each summed in slot order
  const size_t n4 = (size_t)T * d / 4;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i * 4 / d), r = (int)(i * 4 % d);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < K; ++sl) {
      const float4 v = *reinterpret_cast<const float4 *>(p.ys + (size_t)(t * K + sl) * d + r);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    if (p.ns) {
      const float4 v = *reinterpret_cast<const float4 *>(p.ys + (size_t)(T * K + t) * d + r);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    const uint32_t lo = (uint32_t)f32_to_bf16_bits(s.x) | ((uint32_t)f32_to_bf16_bits(s.y) << 16);
    const uint32_t hi = (uint32_t)f32_to_bf16_bits(s.z) | ((uint32_t)f32_to_bf16_bits(s.w) << 16);
    reinterpret_cast<uint2 *>(p.out)[i] = make_uint2(lo, hi);
  }
}

// ---------------------------------------------------------------- tcgen05 contractions
__device__ __forceinline__ void tma2_ef(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                        uint64_t pol) {
  tma_2d_hint(dst, map, x, y, bar, pol);
}
__device__ __forceinline__ void tma2_plain(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// DUAL: gate/up (two weight operands, H = silu(D1) * D2); else down.
template <bool DUAL>
__global__ void __launch_bounds__(kTcThreads, 1) tc_group_kernel(const __grid_constant__ TcParams p) {
  constexpr int kStages = DUAL ? 4 : 6;
  constexpr uint32_t kABytes = kTcM * kTcK * 2;             // 16 KB per weight tile
  constexpr uint32_t kBOff = (DUAL ? 2 : 1) * kABytes;       // token tile after the weight tile(s)
  constexpr uint32_t kStage = kBOff + kTcNMax * kTcK * 2;    // + 16 KB of token rows
  constexpr uint32_t kBuf = (DUAL ? 2 : 1) * kTcNMax;        // TMEM columns of one accumulator buffer
  constexpr uint32_t kCols = 2 * kBuf;                       // two buffers: MMAs of one unit, epilogue of the last
  extern __shared__ __align__(1024) unsigned char tsm_raw[];
  unsigned char *tsm = tsm_raw + ((1024u - (smem_u32(tsm_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long s_full[kStages], s_empty[kStages], s_tfull[2], s_tempty[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_pair[kTcNMax];    // down: pair id of each token column of the unit
  __shared__ float s_wt[kTcNMax];    // down: its routing weight
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(tsm);
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&s_tfull[b]), 1);
      mbar_init(smem_u32(&s_tempty[b]), 4);
    }
    mbar_init(smem_u32(&s_drain), 1);
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the units, tables and token rows come from the previous launches
  const uint32_t tmem = s_tmem;
  const int U = *p.n_units;
  const int nk = p.kdim / kTcK;
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // weights are read once per launch
      int ps = 0, pph = 0, issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const int4 un = p.units[u];
        const int e = p.woken[un.x];
        const int arow = e * p.a_rows + un.y * kTcM;
        const int brow = p.off[un.x] + un.z;
        const int nb = (un.w + kTcBoxN - 1) / kTcBoxN;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait_fast(smem_u32(&s_empty[ps]), pph ^ 1, p.err, DFV_DEVERR_SLOT_WAIT, &s_abort)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&s_full[ps]), dst = sbase + ps * kStage;
          mbar_expect_tx(fb, (uint32_t)((DUAL ? 2 : 1) * kABytes + nb * kTcBoxN * kTcK * 2));
          tma2_ef(dst, &p.tm_a1, kc * kTcK, arow, fb, pol);
          if (DUAL) tma2_ef(dst + kABytes, &p.tm_a2, kc * kTcK, arow, fb, pol);
          for (int j = 0; j < nb; ++j)
            tma2_plain(dst + kBOff + j * (kTcBoxN * kTcK * 2), &p.tm_b, kc * kTcK, brow + j * kTcBoxN, fb);
          ++issued;
          if (++ps == kStages) { ps = 0; pph ^= 1; }
        }
      }
      // no copy may land after the CTA exits: wait for the last fill of every stage
      volatile int never = 0;
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        if (!mbar_wait(smem_u32(&s_full[j % kStages]), (j / kStages) & 1, p.err, DFV_DEVERR_DRAIN_WAIT, &never))
          break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      int cs = 0, cph = 0, tcount = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++tcount) {
        const int4 un = p.units[u];
        const int npad = (un.w + 15) & ~15;
        const uint32_t idesc = idesc_bf16(kTcM, npad);
        const int buf = tcount & 1;
        const uint32_t dbuf = tmem + (uint32_t)buf * kBuf;
        // the epilogue has read this buffer's previous unit (two units ago)
        if (tcount >= 2 && !mbar_wait(smem_u32(&s_tempty[buf]), ((tcount >> 1) - 1) & 1, p.err,
                                      DFV_DEVERR_STAGE_WAIT, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait_fast(smem_u32(&s_full[cs]), cph, p.err, DFV_DEVERR_STAGE_WAIT, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + cs * kStage;
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk) {
            const uint64_t bd = sdesc_k128(st + kBOff) + (uint64_t)(2 * kk);
            const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
            tc_mma(dbuf, sdesc_k128(st) + (uint64_t)(2 * kk), bd, idesc, acc);
            if (DUAL) tc_mma(dbuf + kTcNMax, sdesc_k128(st + kABytes) + (uint64_t)(2 * kk), bd, idesc, acc);
          }
          tc_commit(smem_u32(&s_empty[cs]));  // the stage is free once these MMAs have read it
          if (++cs == kStages) { cs = 0; cph ^= 1; }
        }
        if (ok) tc_commit(smem_u32(&s_tfull[buf]));
      }
      // every MMA issued has completed before TMEM is released
      tc_commit(smem_u32(&s_drain));
      volatile int never = 0;
      mbar_wait(smem_u32(&s_drain), 0u, p.err, DFV_DEVERR_DRAIN_WAIT, &never);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;          // TMEM lanes 32 quad .. 32 quad + 31
    const int row = quad * 32 + lane;   // weight row of the tile this thread reads
    int tcount = 0;
    bool ok = true;
    // after a wait gives up, the loop still runs to the end without touching
    // TMEM, so the four warps meet at every named barrier
    for (int u = blockIdx.x; u < U; u += gridDim.x, ++tcount) {
      const int4 un = p.units[u];
      const int pos0 = p.off[un.x] + un.z;
      if (!DUAL) {
        // the unit's pair ids and weights, fetched while its MMAs run (the
        // previous unit's columns are all stored before they are replaced)
        const int et = tid - 64;  // epilogue thread 0..127
        bar_sync_n(kTcEpiBar, 128);
        if (et < un.w) {
          const int q = p.gather[pos0 + et];
          s_pair[et] = q;
          s_wt[et] = p.w[q];
        }
        bar_sync_n(kTcEpiBar, 128);
      }
      // every lane observes the accumulator barrier itself before it reads TMEM
      const int buf = tcount & 1;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_tfull[buf]), (tcount >> 1) & 1, p.err,
                                                     DFV_DEVERR_STAGE_WAIT, &s_abort));
      if (!ok) continue;
      tc_fence_after();
      const int col = un.y * kTcM + row;  // output column of this thread
      const uint32_t lane_addr = tmem + (uint32_t)buf * kBuf + ((uint32_t)(quad * 32) << 16);
      for (int c0 = 0; c0 < un.w; c0 += 16) {
        float v1[16];
        tmem_ld16(lane_addr + (uint32_t)c0, v1);
        if (DUAL) {
          float v2[16];
          tmem_ld16(lane_addr + kTcNMax + (uint32_t)c0, v2);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < un.w)
              p.h[(size_t)(pos0 + c0 + j) * p.ncols + col] = f32_to_bf16_bits(silu(v1[j]) * v2[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < un.w) p.ys[(size_t)s_pair[c0 + j] * p.ncols + col] = s_wt[c0 + j] * v1[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_tempty[buf]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kCols);
}

template <bool DUAL>
constexpr size_t tc_smem() {
  return 1024 + (size_t)(DUAL ? 4 : 6) * ((DUAL ? 2 : 1) * kTcM * kTcK * 2 + kTcNMax * kTcK * 2);
}

bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by,
                    char *why, size_t why_len) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(why, why_len);
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {bx, by};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(why, why_len, "batched: tensor map encode failed (%d)", (int)r);
    return false;
  }
  return true;
}

template <class Kern, class Par>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Par &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

// Host: the launches of one batched layer, in three phases (0: routing and
// gather, 1: gate/up, 2: down and combine) so that a caller can record events
// between them.  The caller has validated the shapes (bf16, d % 128 == 0,
// d_ff % 128 == 0, d <= 8192, T <= Tmax <= 512).
cudaError_t launch_batch(const BatchParams &p, const dfv_moe_layer *L, int phase, cudaStream_t s, char *why,
                         size_t why_len) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int T = p.T, E = p.E, d = p.d, I = p.I;
  const int P = T * p.K + p.ns * T;
  if (phase == 0) {
    const size_t lsmem = (size_t)kBRowTile * d * 2;
    e = cudaFuncSetAttribute(batch_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lsmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(batch_logits_kernel, dim3((T + kBRowTile - 1) / kBRowTile, (E + kBExpTile - 1) / kBExpTile),
                   dim3(512), lsmem, s, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(batch_topk_kernel, dim3((T + 15) / 16), dim3(512), 0, s, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(batch_tables_kernel, dim3(1), dim3(512), 0, s, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(batch_gather_kernel, dim3(P < 4 * sms ? P : 4 * sms), dim3(256), 0, s, p);
  }
  // contraction tensor maps (weights cached per layer; token maps per workspace)
  TcParams g = {}, dn = {};
  const int Et = E + p.ns;
  if (!encode_bf16_2d(&g.tm_a1, L->w_gate, d, (uint64_t)Et * I, kTcK, kTcM, why, why_len) ||
      !encode_bf16_2d(&g.tm_a2, L->w_up, d, (uint64_t)Et * I, kTcK, kTcM, why, why_len) ||
      !encode_bf16_2d(&g.tm_b, p.xg, d, (uint64_t)P, kTcK, kTcBoxN, why, why_len) ||
      !encode_bf16_2d(&dn.tm_a1, L->w_down, I, (uint64_t)Et * d, kTcK, kTcM, why, why_len) ||
      !encode_bf16_2d(&dn.tm_b, p.h, I, (uint64_t)P, kTcK, kTcBoxN, why, why_len))
    return cudaErrorInvalidValue;
  dn.tm_a2 = dn.tm_a1;
  g.units = p.units_g;
  g.n_units = p.n_units;
  dn.units = p.units_d;
  dn.n_units = p.n_units + 1;
  g.woken = dn.woken = p.woken;
  g.off = dn.off = p.off;
  g.gather = dn.gather = p.gather;
  g.w = dn.w = p.topk_w;
  g.h = dn.h = p.h;
  g.ys = dn.ys = p.ys;
  g.err = dn.err = p.err;
  g.a_rows = I;
  g.kdim = d;
  g.ncols = I;
  dn.a_rows = d;
  dn.kdim = I;
  dn.ncols = d;
  if (phase == 1) {
    e = cudaFuncSetAttribute(tc_group_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem<true>());
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_group_kernel<true>, dim3(sms), dim3(kTcThreads), tc_smem<true>(), s, g);
  }
  e = cudaFuncSetAttribute(tc_group_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc_smem<false>());
  if (e != cudaSuccess) return e;
  e = launch_pdl(tc_group_kernel<false>, dim3(sms), dim3(kTcThreads), tc_smem<false>(), s, dn);
  if (e != cudaSuccess) return e;
  return launch_pdl(batch_combine_kernel, dim3(4 * sms), dim3(256), 0, s, p);
}

}  // namespace dfv
