// dfv_internal.cuh -- device helpers, kernel parameter blocks and the
// workspace layout shared by the kernels of libdfv.so (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dfv.h"

namespace dfv {

constexpr int kMaxBlock = DFV_MAX_BLOCK;
constexpr int kMaxExperts = DFV_MAX_EXPERTS;
constexpr int kMaxTopK = DFV_MAX_TOPK;
constexpr int kDownTile = 64;   // d-rows per down-projection unit (4 warps x 16)
constexpr int kGateTile = 8;    // d_ff rows per gate/up unit (8 gate + 8 up = one m16 tile)

// ---------------------------------------------------------------- workspace
// Every section is 256-byte aligned.  Counters must start at zero; the kernel
// that uses a counter returns it to zero.
//
// Pairs: pair t*K+s is row t's routed slot s; with a shared expert (ns = 1),
// pair k*K+t is row t's shared slot.  The shared expert is the last woken
// expert (id E) and every row selects it, with weight 1.  KS = K + ns.
struct Workspace {
  float *logits;      // [k_max][E]
  int32_t *topk_idx;  // [k_max][K]
  float *topk_w;      // [k_max * KS]  weight of each pair
  int32_t *woken;     // [E + ns]
  int32_t *n_woken;   // [1]           woken experts, the shared one included
  int32_t *offsets;   // [E + ns + 1]
  int32_t *gather;    // [k_max * KS]  pair ids sorted by (expert, t)
  unsigned *router_cnt;  // [1]
  unsigned *err;         // [1] device error bits (DFV_DEVERR_*), sticky until cleared
  unsigned *sync;        // [4] fused kernel: grid-barrier count, exit ticket, abort flag
  unsigned *down_cnt;    // [ceil(d / 16)] one ticket per down tile
  unsigned *flags;       // [1024] mxfp4 single-launch kernel: per-CTA "gate/up work done" flags
  void *xn;           // [k_max][d] activations staged for the expert FFN (act dtype)
  float *h;           // [k_max * KS][d_ff]  SwiGLU activations, by sorted pair position
                      // (bf16 fused kernel: bf16 values, [k*KS][d_ff])
  float *ys;          // [k_max * KS][d]     weighted expert outputs, by pair id
  void *xio;          // [k_max][d] host-variant input staging (4-byte elements)
  void *oio;          // [k_max][d] host-variant output staging
  size_t bytes;
};

// ---------------------------------------------------------------- parameters
struct RouterParams {
  const void *x;        // [k][d] act (input rows; when norm: residual stream)
  const void *wr;       // [E][d]
  int k, d, E, K, norm_topk, act, rdt;
  int ns;               // 1: append the shared expert to the workspace tables
  int fuse_norm;        // 1: route RMSNorm(x) rounded to act, and stage it in ws.xn
  int stage_x;          // 1: copy x into ws.xn (block 0) for the FFN kernels
  float eps;
  Workspace ws;
  // optional user copies of the routing decision
  int32_t *u_idx;
  float *u_w;
  int32_t *u_woken, *u_nw, *u_offs, *u_gather;
};

struct FfnParams {
  // TMA-staged bf16 gate/up: tma_mode 1, one 3-D box per matrix and stage
  // ([ks/64][8 rows][128 B], 128-byte swizzle); 0, one bulk copy per row piece
  CUtensorMap tm_wg, tm_wu, tm_wd;  // tm_wd: down rows [d_ff/64][rs rows][128 B] swizzled
  int tma_mode;
  const void *x;        // [k][d] rows the experts see (bf16 / f32)
  const void *wg, *wu, *wd;
  const uint8_t *sg, *su, *sd;
  const void *residual; // [k][d] or null: added in the combine
  void *out;            // [k][d] act dtype
  int k, d, I, E, K, act;
  int ns;               // 1: the tables end with the shared expert (pairs k*K + t)
  int swz_x;            // XOR swizzle mask for staged x rows (0 or 4)
  int swz_h;            // XOR swizzle mask for staged h rows (0 or 4)
  // TMA-staged kernels only
  int ks;               // TMA gate/up: k-columns per stage slice; mxfp4 gate/up:
                        // parts of d per unit (1, 2 or 4 warps share a row group)
  int nslices;          // gate/up: slices per unit (d / ks)
  int stages;           // ring depth
  int rs;               // down: rows per unit
  Workspace ws;
};

struct FusedParams {
  // block-scaled experts (mxfp4, 8-bit): 2-D tensor maps over the gate / up /
  // down codes (boxes of 64 bytes x 32 or 64 rows, 64-byte swizzle) and the
  // gate / up scales (boxes of 16 bytes x 32 rows); tm_sd over the down scales
  // when a down row takes more than one stage.  The bf16 kernel uses tm_wg and
  // tm_wu for its gate/up boxes.
  CUtensorMap tm_wg, tm_wu, tm_sg, tm_su, tm_wd, tm_sd;
  const void *x;         // [k][d] bf16 rows (the residual stream when fuse_norm)
  const void *residual;  // [k][d] bf16 or null: added in the combine
  void *out;             // [k][d] bf16
  const void *wr, *wg, *wu, *wd;
  const uint8_t *sg, *su, *sd;  // mxfp4 experts: E8M0 scales (null for bf16)
  int k, d, I, E, K, norm_topk, fuse_norm, swz_x;
  int ns;  // 1: one always-on shared expert, id E (pairs k*K + t, weight 1)
  float eps;
  int ks, nsl, slot, scratch, ring;  // filled from the plan
  int tma_mode;  // bf16 gate/up staging: 0 row bulk copies, 1 2-D tensor boxes, 2 one 3-D box per matrix
  Workspace ws;
  int32_t *u_idx, *u_nw;
};

struct FusedPlan {
  int ks, nsl, slot, scratch, ring;
  size_t smem;
};

// One layer of a persistent stack launch (bf16 experts): what changes from
// layer to layer when every layer has the same shape.  The tensor maps sit in
// the kernel parameters, where TMA copies and prefetch.tensormap read them.
struct StackLayer {
  CUtensorMap tm_wg, tm_wu;
  const void *wr, *wg, *wu, *wd;
};
constexpr int kMaxStackLayers = 48;  // layers per launch (parameter space: 48 x 384 bytes)
struct StackParams {
  FusedParams p;  // shape, plan, workspace, the residual stream (x = out = residual)
  int n_layers;
  StackLayer L[kMaxStackLayers];
};

// Batched verify (batch.cu): T = n_blocks * k rows through one bf16 layer.
struct BatchParams {
  const void *x;        // [T][d] bf16 rows
  const void *wr;       // [E][d] bf16 router
  void *out;            // [T][d] bf16
  int T, Tmax, d, E, K, I, ns, norm_topk;
  float *logits;        // [Tmax][E]
  unsigned *tmask;      // [E + 1][Tmax / 32] bit t: row t chose the expert
  int32_t *topk_idx;    // [Tmax][K]
  float *topk_w;        // [Tmax * K + ns * Tmax] pair weights
  int32_t *woken, *off, *n_woken;  // [E + 1], [E + 2], [1]
  int32_t *gather;      // [P] pair ids sorted by (expert, row)
  int *n_units;         // [2] gate/up and down units
  int4 *units_g, *units_d;
  void *xg;             // [P][d] bf16 x rows in sorted order
  uint16_t *h;          // [P][d_ff] bf16
  float *ys;            // [P][d] fp32, by pair id
  unsigned *err;
  int32_t *u_idx, *u_nw;
};

struct AcceptParams {
  const void *logits;   // [k+1][V]
  const int32_t *draft; // [k]
  int32_t *tau, *committed;
  int k, V, dtype, chunks;  // chunks: CTAs per row
  unsigned long long *partial;  // [(k+1) * chunks]
  unsigned *cnt;                // [1]
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 128-bit streaming load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B with fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Load element i of an activation row (bf16 or f32) as float.
__device__ __forceinline__ float load_act(const void *p, size_t i, int act) {
  if (act == DFV_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  return reinterpret_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_act(void *p, size_t i, int act, float v) {
  if (act == DFV_BF16)
    reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(p)[i] = v;
}

// Monotone unsigned key of a float: a < b  <=>  key(a) < key(b), with -0 == +0.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Row of pair q: routed pairs t*K+s, then the shared expert's pairs k*K+t.
__device__ __forceinline__ int pair_token(int q, int k, int K) { return q < k * K ? q / K : q - k * K; }

// ---------------------------------------------------------------- combine
// out[t][r] = residual[t][r] + sum_s ys[t*K+s][r] (slot order) + ys[k*K+t][r]
// (shared expert, when ns) for rows [r0, r0+rows) of every token, by threads
// tid = 0..nthr-1.
__device__ __forceinline__ void combine_rows(const void *residual, void *out, const float *ys, int k, int K, int ns,
                                             int d, int act, int r0, int rows, int tid, int nthr) {
  for (int idx = tid; idx < k * rows; idx += nthr) {
    const int t = idx / rows, r = r0 + idx % rows;
    float s = 0.f;
    for (int sl = 0; sl < K; ++sl) s += __ldcg(ys + (size_t)(t * K + sl) * d + r);
    if (ns) s += __ldcg(ys + (size_t)(k * K + t) * d + r);
    if (residual) s = load_act(residual, (size_t)t * d + r, act) + s;
    store_act(out, (size_t)t * d + r, act, s);
  }
}

// ---------------------------------------------------------------- TMA / mbarrier
constexpr unsigned long long kWaitNs = 2000000000ull;  // bound on any single wait: 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Retire an mbarrier no thread waits on and no copy completes on any more,
// before it is initialised again.
__device__ __forceinline__ void mbar_inval(uint32_t bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `bar` with the given parity.  Gives up when *abort is
// set by another thread of the CTA, or after kWaitNs (then records `code` in
// *err and sets *abort); returns false when it gave up.
static __device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *err, unsigned code,
                                       volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitNs) {
      atomicOr(err, code);
      *abort = 1;
      return false;
    }
  }
}
// mbar_wait with the ready case inlined (no call when the phase is complete).
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, unsigned *err, unsigned code,
                                               volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait(bar, parity, err, code, abort);
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// L2 policy for data read once (streamed weights): evict these lines first,
// so that what is reused across launches (code, router rows, activations,
// routing tables) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// 2-D / 3-D tensor copies global -> shared with an L2 cache policy.
__device__ __forceinline__ void tma_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_3d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}
// Hint: stream `bytes` from global memory into L2 (no completion tracking);
// src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Named barrier over the first n threads of the CTA (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

}  // namespace dfv

// Launch entry points implemented in the .cu files (host side).
namespace dfv {
cudaError_t launch_router(const RouterParams &p, cudaStream_t s, bool pdl);
// phase 0: gate/up, phase 1: down + combine
cudaError_t launch_ffn_phase(const FfnParams &p, int w_dtype, int phase, int grid, cudaStream_t s, bool pdl);
int ffn_grid_limit(int w_dtype, int k, int d, int I, int which);
// mxfp4 experts (ffn_mxfp4.cu): phase 0 = gate/up, 1 = down + combine
int mxfp4_grid_limit(int k, int d, int I, int which);
cudaError_t launch_ffn_mxfp4(const FfnParams &p, int phase, int grid, cudaStream_t s, bool pdl);
// TMA-staged expert FFN: geometry for a layer shape, 0 if it does not fit.
struct TmaPlan {
  int gate_per_sm;  // gate/up CTAs per SM (1 or 2)
  int dsl;          // down stages per unit: 1, or 2 when a stage holds half of d_ff
  int down_per_sm;  // down CTAs per SM (1 or 2)
  int ks, nslices, stages_g, rs, stages_d;
  size_t smem_g, smem_d;
};
bool tma_plan(int w_dtype, int k, int d, int I, TmaPlan *plan);
void ffn_tensor_maps(FfnParams *p, const dfv_moe_layer *L, int ks, int rs, int dsl);
// Fused single-launch layer (bf16): plan, grid (0 = cannot run) and launch.
bool fused_plan(int k, int d, int I, int E, FusedPlan *plan);
int fused_max_grid(const FusedPlan &plan, int k, char *why, size_t why_len);
cudaError_t launch_fused(const FusedParams &p, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl);
int fused_stack_max_grid(const FusedPlan &plan, int k, char *why, size_t why_len);
cudaError_t launch_fused_stack(const StackParams &sp, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl);
bool stack_layer_maps(StackLayer *sl, const dfv_moe_layer *L, const FusedPlan &plan, int max_mode, int *mode);
// fills p->tm_wg / tm_wu and p->tma_mode (<= max_mode) for a bf16 layer (mode 0 when no tensor map fits)
void fused_tensor_maps(FusedParams *p, const dfv_moe_layer *L, const FusedPlan &plan, int max_mode);
// single-launch layer with block-scaled experts, fmt = DFV_MXFP4 or DFV_Q8
// (layer_fused_bs.cu)
bool fused_bs_plan(int fmt, int k, int d, int I, int E, FusedPlan *plan);
// fills p->tm_* for a block-scaled layer; false (with a reason) when the driver refuses
bool fused_bs_tensor_maps(FusedParams *p, const dfv_moe_layer *L, char *why, size_t why_len);
int fused_bs_max_grid(const FusedPlan &plan, int fmt, int k, char *why, size_t why_len);
cudaError_t launch_fused_bs(const FusedParams &p, int fmt, const FusedPlan &plan, int grid, cudaStream_t s, bool pdl);
// phase 0 gate/up, 1 down (writes ys), 2 combine
cudaError_t launch_ffn_tma(const FfnParams &p, int w_dtype, int phase, const TmaPlan &plan, int grid, cudaStream_t s,
                           bool pdl);
cudaError_t launch_accept(const AcceptParams &p, cudaStream_t s);
// batched verify (batch.cu), phase 0 routing + gather, 1 gate/up, 2 down + combine;
// `why` receives a reason when a tensor map cannot be built
cudaError_t launch_batch(const BatchParams &p, const dfv_moe_layer *L, int phase, cudaStream_t s, char *why,
                         size_t why_len);
// device address of the fixed acceptance scratch array on the current device
cudaError_t accept_noalloc_scratch(void **out);
int accept_noalloc_max_chunks();
}  // namespace dfv
