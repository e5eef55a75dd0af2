// api.cu -- the C ABI of libdfv.so: argument validation, workspace layout and
// launch order.  Every entry point validates on the host, then only enqueues
// kernels (and, for the host-buffer variant, copies) on the caller's stream.
#include <mutex>
#include <map>
#include <string>
#include <tuple>
#include <cstdarg>
#include <cstdio>

#include "dfv_internal.cuh"

namespace dfv {
cudaError_t launch_wait_selftest(const Workspace &w, cudaStream_t s);  // selftest.cu
cudaError_t launch_mma_selftest(const void *A, const void *B, float *D, int bf16, cudaStream_t s);
cudaError_t launch_tc05_selftest(const void *A, const void *B, int N, int K, float *D, int *status, cudaStream_t s);
}

namespace {

thread_local std::string g_detail;
thread_local cudaEvent_t g_events[4];
thread_local bool g_profile = false;
thread_local int g_last_path = -1;
std::string g_fused_why;  // why the fused path is unavailable (first failure)
thread_local int g_max_staging = 3;   // highest gate/up staging mode of the bf16 fused kernel
thread_local int g_last_staging = -1;

inline void mark(int i, cudaStream_t s) {
  if (g_profile) cudaEventRecord(g_events[i], s);
}

int fail(int status, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char *where) {
  return fail(DFV_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t act_size(int act) { return act == DFV_BF16 ? 2 : 4; }

// Workspace sections, in order; base == nullptr only measures.
dfv::Workspace layout(const dfv_moe_layer *L, int k_max, void *base) {
  dfv::Workspace w = {};
  const size_t E = L->n_experts, K = L->top_k, d = L->d, I = L->d_ff, km = k_max;
  const size_t ns = L->n_shared ? 1 : 0, KS = K + ns;  // pair slots per row: routed, then shared
  size_t off = 0;
  auto take = [&](size_t bytes) -> void * {
    void *p = base ? (void *)((char *)base + off) : nullptr;
    off += align256(bytes);
    return p;
  };
  // counters and the error word first, at offsets that depend on nothing but d
  // (a fixed 8 KB for d <= 13312): calls of any k, and layers of any width in
  // that range, can share a workspace
  w.router_cnt = (unsigned *)take(4);
  w.err = (unsigned *)take(4);
  w.sync = (unsigned *)take(16);
  const size_t tiles = (d + 15) / 16;
  w.down_cnt = (unsigned *)take(tiles * 4 > 3328 ? tiles * 4 : 3328);
  w.flags = (unsigned *)take(1024 * 4);
  w.logits = (float *)take(km * E * 4);
  w.topk_idx = (int32_t *)take(km * K * 4);
  w.topk_w = (float *)take(km * KS * 4);
  w.woken = (int32_t *)take((E + ns) * 4);
  w.n_woken = (int32_t *)take(4);
  w.offsets = (int32_t *)take((E + ns + 1) * 4);
  w.gather = (int32_t *)take(km * KS * 4);
  w.xn = take(km * d * 4);
  w.h = (float *)take(km * KS * I * 4);
  w.ys = (float *)take(km * KS * d * 4);
  w.xio = take(km * d * 4);
  w.oio = take(km * d * 4);
  w.bytes = off;
  return w;
}

int check_layer(const dfv_moe_layer *L, int act) {
  if (!L) return fail(DFV_ERR_INVALID_ARG, "layer is NULL");
  if (L->d <= 0 || L->n_experts <= 0 || L->top_k <= 0 || L->d_ff <= 0)
    return fail(DFV_ERR_INVALID_ARG, "non-positive layer size");
  if (L->n_experts > DFV_MAX_EXPERTS) return fail(DFV_ERR_UNSUPPORTED, "n_experts %d > %d", L->n_experts, DFV_MAX_EXPERTS);
  if (L->top_k > DFV_MAX_TOPK || L->top_k > L->n_experts)
    return fail(DFV_ERR_UNSUPPORTED, "top_k %d outside 1..min(E, %d)", L->top_k, DFV_MAX_TOPK);
  if (L->n_shared < 0) return fail(DFV_ERR_INVALID_ARG, "n_shared %d < 0", L->n_shared);
  if (L->n_shared > 1) return fail(DFV_ERR_UNSUPPORTED, "n_shared %d > 1", L->n_shared);
  if (L->d % 32 || L->d_ff % 32) return fail(DFV_ERR_UNSUPPORTED, "d and d_ff must be multiples of 32");
  const bool ok = (L->w_dtype == DFV_BF16 && L->r_dtype == DFV_BF16 && act == DFV_BF16) ||
                  (L->w_dtype == DFV_MXFP4 && L->r_dtype == DFV_BF16 && act == DFV_BF16) ||
                  (L->w_dtype == DFV_Q8 && L->r_dtype == DFV_BF16 && act == DFV_BF16) ||
                  (L->w_dtype == DFV_F32 && L->r_dtype == DFV_F32 && act == DFV_F32);
  if (!ok)
    return fail(DFV_ERR_UNSUPPORTED, "unsupported dtype combination (experts %d, router %d, act %d)", L->w_dtype,
                L->r_dtype, act);
  if (!L->w_router || !L->w_gate || !L->w_up || !L->w_down) return fail(DFV_ERR_INVALID_ARG, "NULL weight pointer");
  if (L->w_dtype == DFV_MXFP4 || L->w_dtype == DFV_Q8) {
    if (L->w_dtype == DFV_MXFP4 && (L->d % 64 || L->d_ff % 64))
      return fail(DFV_ERR_UNSUPPORTED, "mxfp4 layers need d and d_ff multiples of 64");
    if (L->w_dtype == DFV_Q8) {
      dfv::FusedPlan qp;
      if (!dfv::fused_bs_plan(DFV_Q8, 1, L->d, L->d_ff, L->n_experts, &qp))
        return fail(DFV_ERR_UNSUPPORTED, "8-bit layers need d %% 256 == 0, d <= 2048, d_ff %% 64 == 0, "
                                         "64 <= d_ff <= 512 and d_ff %% 256 == 0 above 256 (d=%d, d_ff=%d)",
                    L->d, L->d_ff);
    }
    if (!L->s_gate || !L->s_up || !L->s_down) return fail(DFV_ERR_INVALID_ARG, "block-scaled layer without scale pointers");
    if (!aligned(L->s_gate, 16) || !aligned(L->s_up, 16) || !aligned(L->s_down, 16))
      return fail(DFV_ERR_INVALID_ARG, "scale pointers must be 16-byte aligned");
  }
  if (!aligned(L->w_router, 16) || !aligned(L->w_gate, 16) || !aligned(L->w_up, 16) || !aligned(L->w_down, 16))
    return fail(DFV_ERR_INVALID_ARG, "weight pointers must be 16-byte aligned");
  return DFV_OK;
}

int check_ws(const dfv_moe_layer *L, int k, void *ws, size_t ws_bytes) {
  if (!ws) return fail(DFV_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(DFV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const size_t need = layout(L, k, nullptr).bytes;
  if (ws_bytes < need) return fail(DFV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  return DFV_OK;
}

// Occupancy-limited persistent grid sizes, cached per (dtype, k<=8, d, I, which).
int grid_limit(int w_dtype, int k, int d, int I, int which) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  auto key = std::make_tuple(dev, w_dtype, k <= 8 ? 1 : 2, d, I, which);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int g = dfv::ffn_grid_limit(w_dtype, k, d, I, which);
  if (g > 0) cache[key] = g;
  return g;
}

int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = n;
  return n;
}

dfv::RouterParams router_params(const dfv_moe_layer *L, const void *x, int act, int k, const dfv::Workspace &w) {
  dfv::RouterParams p = {};
  p.x = x;
  p.wr = L->w_router;
  p.k = k;
  p.d = L->d;
  p.E = L->n_experts;
  p.K = L->top_k;
  p.norm_topk = L->norm_topk ? 1 : 0;
  p.ns = L->n_shared ? 1 : 0;
  p.act = act;
  p.rdt = L->r_dtype;
  p.ws = w;
  return p;
}

// Single-launch fused layer (bf16 or mxfp4 experts): grid = SM count, cooperative.
// Returns -1 when the shape or the device does not allow it (the caller then
// uses the multi-kernel path), else a DFV status.
int run_layer_fused(const dfv_moe_layer *L, const void *x, int act, int k, void *out, const void *residual,
                    bool fuse_norm, float eps, int32_t *u_idx, int32_t *u_nw, const dfv::Workspace &w,
                    cudaStream_t s) {
  const bool mx = L->w_dtype == DFV_MXFP4 || L->w_dtype == DFV_Q8;  // block-scaled experts
  if ((L->w_dtype != DFV_BF16 && !mx) || L->r_dtype != DFV_BF16 || act != DFV_BF16) return -1;
  dfv::FusedPlan plan;
  if (!(mx ? dfv::fused_bs_plan(L->w_dtype, k, L->d, L->d_ff, L->n_experts, &plan)
           : dfv::fused_plan(k, L->d, L->d_ff, L->n_experts, &plan)))
    return -1;
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  int grid;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(dev, mx ? L->w_dtype : 0, k <= 8 ? 1 : 2, plan.smem);
    auto it = cache.find(key);
    if (it == cache.end()) {
      char why[256] = {0};
      const int gmax = mx ? dfv::fused_bs_max_grid(plan, L->w_dtype, k, why, sizeof why)
                          : dfv::fused_max_grid(plan, k, why, sizeof why);
      if (gmax <= 0 && g_fused_why.empty()) g_fused_why = why;
      it = cache.emplace(key, gmax).first;
    }
    grid = it->second;
  }
  if (grid <= 0) return -1;
  dfv::FusedParams fp = {};
  fp.x = x;
  fp.residual = residual;
  fp.out = out;
  fp.wr = L->w_router;
  fp.wg = L->w_gate;
  fp.wu = L->w_up;
  fp.wd = L->w_down;
  if (mx) {
    fp.sg = L->s_gate;
    fp.su = L->s_up;
    fp.sd = L->s_down;
    char why[256] = {0};
    if (!dfv::fused_bs_tensor_maps(&fp, L, why, sizeof why)) {
      std::lock_guard<std::mutex> lock(mu);
      if (g_fused_why.empty()) g_fused_why = why;
      return -1;
    }
  }
  fp.k = k;
  fp.d = L->d;
  fp.I = L->d_ff;
  fp.E = L->n_experts;
  fp.K = L->top_k;
  fp.norm_topk = L->norm_topk ? 1 : 0;
  fp.ns = L->n_shared ? 1 : 0;
  fp.fuse_norm = fuse_norm ? 1 : 0;
  fp.swz_x = (L->d % 64 == 0) ? 4 : 0;
  fp.eps = eps;
  fp.ws = w;
  fp.u_idx = u_idx;
  fp.u_nw = u_nw;
  if (!mx) {
    dfv::fused_tensor_maps(&fp, L, plan, g_max_staging);
    g_last_staging = fp.tma_mode;
  }
  auto go = [&](bool pdl) {
    return mx ? dfv::launch_fused_bs(fp, L->w_dtype, plan, grid, s, pdl) : dfv::launch_fused(fp, plan, grid, s, pdl);
  };
  mark(0, s);
  cudaError_t e = go(true);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear, and retry without programmatic serialisation
    e = go(false);
  }
  if (e != cudaSuccess) return cuda_fail(e, "fused layer launch");
  mark(1, s);
  mark(2, s);
  mark(3, s);
  return DFV_OK;
}

// Batched-verify workspace: counters (first 256 bytes), the error word at byte
// 256 (as in the single-block workspace), then the tables and buffers.
struct BatchWs {
  dfv::BatchParams p;
  size_t bytes;
};
BatchWs batch_layout(const dfv_moe_layer *L, int tmax, void *base) {
  BatchWs b = {};
  const size_t E = L->n_experts, K = L->top_k, d = L->d, I = L->d_ff, ns = L->n_shared ? 1 : 0;
  const size_t T = ((size_t)tmax + 31) / 32 * 32, P = T * K + ns * T;
  // units: per woken expert, row tiles x passes of <= 128 tokens; the passes
  // over all experts number at most (E + 1) + P / 128
  const size_t units = ((E + 1) + P / 128 + 1) * ((I > d ? I : d) / 128);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void * {
    void *q = base ? (void *)((char *)base + off) : nullptr;
    off += align256(bytes);
    return q;
  };
  b.p.n_units = (int *)take(16);
  b.p.err = (unsigned *)take(4);
  b.p.n_woken = (int32_t *)take(4);
  b.p.logits = (float *)take(T * E * 4);
  b.p.tmask = (unsigned *)take((E + 1) * (T / 32) * 4);
  b.p.topk_idx = (int32_t *)take(T * K * 4);
  b.p.topk_w = (float *)take(P * 4);
  b.p.woken = (int32_t *)take((E + 1) * 4);
  b.p.off = (int32_t *)take((E + 2) * 4);
  b.p.gather = (int32_t *)take(P * 4);
  b.p.units_g = (int4 *)take(units * 16);
  b.p.units_d = (int4 *)take(units * 16);
  b.p.xg = take(P * d * 2);
  b.p.h = (uint16_t *)take(P * I * 2);
  b.p.ys = (float *)take(P * d * 4);
  b.p.Tmax = (int)T;
  b.bytes = off;
  return b;
}

thread_local bool g_fused_enabled = true;
thread_local int g_stack_mode = 1;  // 0 per layer, 1 persistent for eager calls with k <= 8, 2 persistent

// A residual stack of bf16 layers of one shape as persistent launches of up
// to kMaxStackLayers layers each.  Returns -1 when the layers or the device do
// not allow it (the caller then launches layer by layer), else a DFV status.
int run_stack_persistent(const dfv_moe_layer *Ls, int n_layers, void *x, int k, float eps, int32_t *u_nw,
                         void *ws, cudaStream_t s) {
  const dfv_moe_layer &L0 = Ls[0];
  for (int l = 0; l < n_layers; ++l) {
    const dfv_moe_layer &L = Ls[l];
    if (L.w_dtype != DFV_BF16 || L.r_dtype != DFV_BF16 || L.d != L0.d || L.d_ff != L0.d_ff ||
        L.n_experts != L0.n_experts || L.top_k != L0.top_k || (L.n_shared != 0) != (L0.n_shared != 0) ||
        (L.norm_topk != 0) != (L0.norm_topk != 0))
      return -1;
  }
  dfv::FusedPlan plan;
  if (!dfv::fused_plan(k, L0.d, L0.d_ff, L0.n_experts, &plan)) return -1;
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  int grid;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(dev, k <= 8 ? 1 : 2, plan.smem);
    auto it = cache.find(key);
    if (it == cache.end()) {
      char why[256] = {0};
      const int gmax = dfv::fused_stack_max_grid(plan, k, why, sizeof why);
      if (gmax <= 0 && g_fused_why.empty()) g_fused_why = why;
      it = cache.emplace(key, gmax).first;
    }
    grid = it->second;
  }
  if (grid <= 0) return -1;
  // the parameter block carries every layer's tensor maps
  static thread_local dfv::StackParams sp;
  sp = dfv::StackParams{};
  dfv::FusedParams &fp = sp.p;
  fp.x = x;
  fp.residual = x;
  fp.out = x;
  fp.k = k;
  fp.d = L0.d;
  fp.I = L0.d_ff;
  fp.E = L0.n_experts;
  fp.K = L0.top_k;
  fp.norm_topk = L0.norm_topk ? 1 : 0;
  fp.ns = L0.n_shared ? 1 : 0;
  fp.fuse_norm = 1;
  fp.swz_x = (L0.d % 64 == 0) ? 4 : 0;
  fp.eps = eps;
  fp.ws = layout(&L0, k, ws);
  for (int l0 = 0; l0 < n_layers; l0 += dfv::kMaxStackLayers) {
    const int n = n_layers - l0 < dfv::kMaxStackLayers ? n_layers - l0 : dfv::kMaxStackLayers;
    // every layer of a launch takes the same staging mode: the lowest any
    // layer's maps allow
    int mode = g_max_staging;
    for (int pass = 0; pass < 2; ++pass) {
      int lo = mode;
      for (int i = 0; i < n; ++i) {
        int m = 0;
        dfv::stack_layer_maps(&sp.L[i], &Ls[l0 + i], plan, mode, &m);
        lo = m < lo ? m : lo;
      }
      if (lo == mode) break;
      mode = lo;
    }
    fp.tma_mode = mode;
    fp.u_nw = u_nw ? u_nw + l0 : nullptr;
    g_last_staging = mode;
    sp.n_layers = n;
    mark(0, s);
    cudaError_t e = dfv::launch_fused_stack(sp, plan, grid, s, true);
    if (e != cudaSuccess) {
      cudaGetLastError();
      e = dfv::launch_fused_stack(sp, plan, grid, s, false);
    }
    if (e != cudaSuccess) return cuda_fail(e, "persistent stack launch");
    mark(1, s);
    mark(2, s);
    mark(3, s);
  }
  g_last_path = 3;
  return DFV_OK;
}

int run_layer(const dfv_moe_layer *L, const void *x, int act, int k, void *out, const void *residual,
              bool fuse_norm, float eps, int32_t *u_idx, int32_t *u_nw, const dfv::Workspace &w, cudaStream_t s) {
  if (g_fused_enabled) {
    const int st = run_layer_fused(L, x, act, k, out, residual, fuse_norm, eps, u_idx, u_nw, w, s);
    if (st >= 0) {
      g_last_path = 1;
      return st;
    }
  }
  if (L->w_dtype == DFV_Q8)  // 8-bit weights run only in the single-launch kernel
    return fail(DFV_ERR_UNSUPPORTED, "8-bit layer: the single-launch kernel is unavailable (%s)",
                g_fused_enabled ? g_fused_why.c_str() : "multi-kernel path selected");
  g_last_path = 0;
  dfv::RouterParams rp = router_params(L, x, act, k, w);
  rp.fuse_norm = fuse_norm ? 1 : 0;
  rp.eps = eps;
  rp.u_idx = u_idx;
  rp.u_nw = u_nw;
  mark(0, s);
  cudaError_t e = dfv::launch_router(rp, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  mark(1, s);

  dfv::FfnParams fp = {};
  fp.x = fuse_norm ? w.xn : x;
  fp.wg = L->w_gate;
  fp.wu = L->w_up;
  fp.wd = L->w_down;
  fp.sg = L->s_gate;
  fp.su = L->s_up;
  fp.sd = L->s_down;
  fp.residual = residual;
  fp.out = out;
  fp.k = k;
  fp.d = L->d;
  fp.I = L->d_ff;
  fp.E = L->n_experts;
  fp.K = L->top_k;
  fp.ns = L->n_shared ? 1 : 0;
  fp.act = act;
  fp.swz_x = (L->d % 64 == 0) ? 4 : 0;
  fp.swz_h = (L->d_ff % 64 == 0) ? 4 : 0;
  fp.ws = w;
  const int maxW = (L->n_experts < k * L->top_k ? L->n_experts : k * L->top_k) + fp.ns;  // + the shared expert
  if (L->w_dtype == DFV_MXFP4) {
    // codes widened in registers: gate/up units of (expert, 8 * 4/ks rows),
    // ks the smallest split of d whose units still fill two CTAs per SM.  ks
    // sets how each row's sum splits over d, so it is chosen for the largest
    // block and is the same for every k (a block's rows then equal
    // single-token calls bit for bit)
    const int sms = sm_count();
    if (sms <= 0) return fail(DFV_ERR_CUDA, "cannot query the SM count");
    const int maxW16 = (L->n_experts < DFV_MAX_BLOCK * L->top_k ? L->n_experts : DFV_MAX_BLOCK * L->top_k) + fp.ns;
    int ks = 1;
    while (ks < 4 && maxW16 * (L->d_ff / (8 * (4 / ks))) < 2 * sms) ks *= 2;
    fp.ks = ks;
    const int units_g = maxW * (L->d_ff / (8 * (4 / ks)));
    const int units_d = maxW * (L->d / dfv::kDownTile);
    const int lim_g = grid_limit(L->w_dtype, k, L->d, L->d_ff, 0);
    const int lim_d = grid_limit(L->w_dtype, k, L->d, L->d_ff, 1);
    if (lim_g <= 0 || lim_d <= 0) return fail(DFV_ERR_CUDA, "mxfp4 expert kernels cannot be resident (occupancy 0)");
    e = dfv::launch_ffn_mxfp4(fp, 0, units_g < lim_g ? units_g : lim_g, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "mxfp4 expert gate/up launch");
    mark(2, s);
    e = dfv::launch_ffn_mxfp4(fp, 1, units_d < lim_d ? units_d : lim_d, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "mxfp4 expert down/combine launch");
    mark(3, s);
    return DFV_OK;
  }
  dfv::TmaPlan plan;
  if (dfv::tma_plan(L->w_dtype, k, L->d, L->d_ff, &plan)) {
    // TMA-staged kernels: one persistent CTA per SM
    const int sms = sm_count();
    if (sms <= 0) return fail(DFV_ERR_CUDA, "cannot query the SM count");
    const int units_g = maxW * (L->d_ff / dfv::kGateTile);
    const int units_d = maxW * ((L->d + plan.rs - 1) / plan.rs);
    if (g_max_staging > 0) dfv::ffn_tensor_maps(&fp, L, plan.ks, plan.rs, plan.dsl);  // else mode 0: bulk copies
    const int gg = plan.gate_per_sm * sms;
    e = dfv::launch_ffn_tma(fp, L->w_dtype, 0, plan, units_g < gg ? units_g : gg, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "expert gate/up launch");
    mark(2, s);
    const int gd = plan.down_per_sm * sms;
    e = dfv::launch_ffn_tma(fp, L->w_dtype, 1, plan, units_d < gd ? units_d : gd, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "expert down launch");
    e = dfv::launch_ffn_tma(fp, L->w_dtype, 2, plan, sms, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    mark(3, s);
    return DFV_OK;
  }
  const int units_g = maxW * (L->d_ff / dfv::kGateTile);
  const int units_d = maxW * ((L->d + dfv::kDownTile - 1) / dfv::kDownTile);
  const int lim_g = grid_limit(L->w_dtype, k, L->d, L->d_ff, 0);
  const int lim_d = grid_limit(L->w_dtype, k, L->d, L->d_ff, 1);
  if (lim_g <= 0 || lim_d <= 0) return fail(DFV_ERR_CUDA, "expert FFN kernels cannot be resident (occupancy 0)");
  const int gg = units_g < lim_g ? units_g : lim_g;
  const int gd = units_d < lim_d ? units_d : lim_d;
  e = dfv::launch_ffn_phase(fp, L->w_dtype, 0, gg, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "expert gate/up launch");
  mark(2, s);
  e = dfv::launch_ffn_phase(fp, L->w_dtype, 1, gd, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "expert down/combine launch");
  mark(3, s);
  return DFV_OK;
}

}  // namespace

extern "C" {

int dfv_version(void) { return DFV_VERSION; }

const char *dfv_status_string(int status) {
  switch (status) {
    case DFV_OK: return "DFV_OK";
    case DFV_ERR_INVALID_ARG: return "DFV_ERR_INVALID_ARG";
    case DFV_ERR_UNSUPPORTED: return "DFV_ERR_UNSUPPORTED";
    case DFV_ERR_WORKSPACE: return "DFV_ERR_WORKSPACE";
    case DFV_ERR_CUDA: return "DFV_ERR_CUDA";
    default: return "DFV_ERR_UNKNOWN";
  }
}

const char *dfv_last_error_detail(void) { return g_detail.c_str(); }

int dfv_profile_set_events(void *const *events, int n_events) {
  if (!events) {
    g_profile = false;
    return DFV_OK;
  }
  if (n_events < 4) return fail(DFV_ERR_INVALID_ARG, "need 4 events, got %d", n_events);
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return fail(DFV_ERR_INVALID_ARG, "event %d is NULL", i);
    g_events[i] = (cudaEvent_t)events[i];
  }
  g_profile = true;
  return DFV_OK;
}

size_t dfv_moe_workspace_size(const dfv_moe_layer *layer, int k_max) {
  if (!layer || k_max < 1 || k_max > DFV_MAX_BLOCK || layer->n_experts <= 0 || layer->top_k <= 0 ||
      layer->d <= 0 || layer->d_ff <= 0 || layer->n_shared < 0 || layer->n_shared > 1)
    return 0;
  return layout(layer, k_max, nullptr).bytes;
}

int dfv_route_topk(const dfv_moe_layer *layer, const void *hidden, int act, int k, int32_t *topk_idx,
                   float *topk_w, int32_t *woken, int32_t *n_woken, int32_t *offsets, int32_t *gather, void *ws,
                   size_t ws_bytes, void *stream) {
  int st = check_layer(layer, act);
  if (st) return st;
  if (k < 1 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 1..%d", k, DFV_MAX_BLOCK);
  if (!hidden || !aligned(hidden, 16)) return fail(DFV_ERR_INVALID_ARG, "hidden NULL or not 16-byte aligned");
  if (!n_woken) return fail(DFV_ERR_INVALID_ARG, "n_woken is NULL");
  if ((st = check_ws(layer, k, ws, ws_bytes))) return st;
  const dfv::Workspace w = layout(layer, k, ws);
  dfv::RouterParams rp = router_params(layer, hidden, act, k, w);
  rp.u_idx = topk_idx;
  rp.u_w = topk_w;
  rp.u_woken = woken;
  rp.u_nw = n_woken;
  rp.u_offs = offsets;
  rp.u_gather = gather;
  cudaError_t e = dfv::launch_router(rp, (cudaStream_t)stream, true);
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  return DFV_OK;
}

int dfv_moe_block_forward(const dfv_moe_layer *layer, const void *hidden, int act, int k, void *out,
                          int32_t *opt_topk_idx, int32_t *opt_n_woken, void *ws, size_t ws_bytes, void *stream) {
  int st = check_layer(layer, act);
  if (st) return st;
  if (k < 1 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 1..%d", k, DFV_MAX_BLOCK);
  if (!hidden || !out || !aligned(hidden, 16) || !aligned(out, 16))
    return fail(DFV_ERR_INVALID_ARG, "hidden/out NULL or not 16-byte aligned");
  if ((st = check_ws(layer, k, ws, ws_bytes))) return st;
  const dfv::Workspace w = layout(layer, k, ws);
  return run_layer(layer, hidden, act, k, out, nullptr, false, 0.f, opt_topk_idx, opt_n_woken, w,
                   (cudaStream_t)stream);
}

int dfv_moe_block_forward_host(const dfv_moe_layer *layer, const void *hidden_host, int act, int k, void *out_host,
                               void *ws, size_t ws_bytes, void *stream) {
  int st = check_layer(layer, act);
  if (st) return st;
  if (k < 1 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 1..%d", k, DFV_MAX_BLOCK);
  if (!hidden_host || !out_host) return fail(DFV_ERR_INVALID_ARG, "host buffers must not be NULL");
  if ((st = check_ws(layer, k, ws, ws_bytes))) return st;
  const dfv::Workspace w = layout(layer, k, ws);
  const size_t bytes = (size_t)k * layer->d * act_size(act);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(w.xio, hidden_host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "host->device copy of hidden");
  if ((st = run_layer(layer, w.xio, act, k, w.oio, nullptr, false, 0.f, nullptr, nullptr, w, s))) return st;
  e = cudaMemcpyAsync(out_host, w.oio, bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "device->host copy of out");
  return DFV_OK;
}

int dfv_moe_stack_forward(const dfv_moe_layer *layers, int n_layers, void *x, int k, float eps,
                          int32_t *opt_n_woken, void *ws, size_t ws_bytes, void *stream) {
  if (!layers || n_layers < 1) return fail(DFV_ERR_INVALID_ARG, "no layers");
  if (k < 1 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 1..%d", k, DFV_MAX_BLOCK);
  if (!x || !aligned(x, 16)) return fail(DFV_ERR_INVALID_ARG, "x NULL or not 16-byte aligned");
  if (!(eps >= 0.f)) return fail(DFV_ERR_INVALID_ARG, "eps must be >= 0");
  for (int l = 0; l < n_layers; ++l) {
    int st = check_layer(&layers[l], DFV_BF16);
    if (st) return fail(st, "layer %d: %s", l, g_detail.c_str());
    if (layers[l].d != layers[0].d) return fail(DFV_ERR_INVALID_ARG, "layer %d: d differs from layer 0", l);
    if ((st = check_ws(&layers[l], k, ws, ws_bytes))) return fail(st, "layer %d: %s", l, g_detail.c_str());
  }
  bool persistent = g_stack_mode == 2;
  if (g_stack_mode == 1 && k <= 8) {
    // measured: inside a CUDA graph, per-layer launches chained programmatically
    // are faster than the persistent kernel's layer-boundary grid barrier
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    persistent = cudaStreamIsCapturing((cudaStream_t)stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone;
  }
  if (g_fused_enabled && persistent) {
    const int st = run_stack_persistent(layers, n_layers, x, k, eps, opt_n_woken, ws, (cudaStream_t)stream);
    if (st >= 0) return st;
  }
  for (int l = 0; l < n_layers; ++l) {
    const dfv::Workspace w = layout(&layers[l], k, ws);
    int st = run_layer(&layers[l], x, DFV_BF16, k, x, x, true, eps, nullptr, opt_n_woken ? opt_n_woken + l : nullptr,
                       w, (cudaStream_t)stream);
    if (st) return st;
  }
  return DFV_OK;
}

size_t dfv_moe_batch_workspace_size(const dfv_moe_layer *layer, int n_rows_max) {
  if (!layer || n_rows_max < 1 || n_rows_max > DFV_MAX_BATCH_ROWS || layer->n_experts <= 0 || layer->top_k <= 0 ||
      layer->d <= 0 || layer->d_ff <= 0 || layer->n_shared < 0 || layer->n_shared > 1)
    return 0;
  return batch_layout(layer, n_rows_max, nullptr).bytes;
}

int dfv_moe_batch_forward(const dfv_moe_layer *layer, const void *hidden, int n_blocks, int k, void *out,
                          int32_t *opt_topk_idx, int32_t *opt_n_woken, void *ws, size_t ws_bytes, void *stream) {
  int st = check_layer(layer, DFV_BF16);
  if (st) return st;
  if (layer->w_dtype != DFV_BF16) return fail(DFV_ERR_UNSUPPORTED, "batched verify takes bf16 expert weights");
  if (layer->d % 128 || layer->d_ff % 128 || layer->d > 8192)
    return fail(DFV_ERR_UNSUPPORTED, "batched verify needs d and d_ff multiples of 128 and d <= 8192 (d=%d, d_ff=%d)",
                layer->d, layer->d_ff);
  if (k < 1 || k > DFV_MAX_BLOCK || n_blocks < 1 || n_blocks * k > DFV_MAX_BATCH_ROWS)
    return fail(DFV_ERR_INVALID_ARG, "n_blocks=%d, k=%d: need 1 <= k <= %d and n_blocks * k <= %d", n_blocks, k,
                DFV_MAX_BLOCK, DFV_MAX_BATCH_ROWS);
  if (!hidden || !out || !aligned(hidden, 16) || !aligned(out, 16))
    return fail(DFV_ERR_INVALID_ARG, "hidden/out NULL or not 16-byte aligned");
  if (!ws || !aligned(ws, 256)) return fail(DFV_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  const int T = n_blocks * k;
  const size_t need = batch_layout(layer, T, nullptr).bytes;
  if (ws_bytes < need) return fail(DFV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  BatchWs b = batch_layout(layer, T, ws);
  dfv::BatchParams &p = b.p;
  p.x = hidden;
  p.wr = layer->w_router;
  p.out = out;
  p.T = T;
  p.d = layer->d;
  p.E = layer->n_experts;
  p.K = layer->top_k;
  p.I = layer->d_ff;
  p.ns = layer->n_shared ? 1 : 0;
  p.norm_topk = layer->norm_topk ? 1 : 0;
  p.u_idx = opt_topk_idx;
  p.u_nw = opt_n_woken;
  char why[256] = {0};
  cudaStream_t s = (cudaStream_t)stream;
  mark(0, s);
  for (int phase = 0; phase < 3; ++phase) {
    cudaError_t e = dfv::launch_batch(p, layer, phase, s, why, sizeof why);
    if (e != cudaSuccess) {
      if (why[0]) return fail(DFV_ERR_CUDA, "batched verify: %s", why);
      return cuda_fail(e, "batched verify launch");
    }
    mark(phase + 1, s);
  }
  g_last_path = 2;
  return DFV_OK;
}

int dfv_last_layer_path(void) { return g_last_path; }

const char *dfv_fused_unavailable_reason(void) { return g_fused_why.c_str(); }

int dfv_set_staging(int max_mode) {
  if (max_mode < 0 || max_mode > 3) return fail(DFV_ERR_INVALID_ARG, "staging mode must be 0, 1, 2 or 3");
  g_max_staging = max_mode;
  return DFV_OK;
}

int dfv_last_staging(void) { return g_last_staging; }

int dfv_set_stack_launch(int mode) {
  if (mode < 0 || mode > 2) return fail(DFV_ERR_INVALID_ARG, "stack launch mode must be 0, 1 or 2");
  g_stack_mode = mode;
  return DFV_OK;
}

int dfv_set_path(int path) {
  if (path != 0 && path != 1) return fail(DFV_ERR_INVALID_ARG, "path must be 0 (multi-kernel) or 1 (fused)");
  g_fused_enabled = path == 1;
  return DFV_OK;
}

int dfv_selftest_bounded_waits(void *ws, size_t ws_bytes, void *stream) {
  if (!ws) return fail(DFV_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(DFV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  // the counters sit at fixed offsets, the same for every layer up to d = 13312
  dfv_moe_layer probe = {};
  probe.d = 32;
  probe.n_experts = 1;
  probe.top_k = 1;
  probe.d_ff = 32;
  const size_t need = layout(&probe, 1, nullptr).bytes;
  if (ws_bytes < need) return fail(DFV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  cudaError_t e = dfv::launch_wait_selftest(layout(&probe, 1, ws), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test launch");
  return DFV_OK;
}

int dfv_selftest_mma(int dtype, const void *A, const void *B, float *D, void *stream) {
  if (dtype != DFV_BF16 && dtype != DFV_F16) return fail(DFV_ERR_UNSUPPORTED, "MMA self-test dtype %d", dtype);
  if (!A || !B || !D || !aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
    return fail(DFV_ERR_INVALID_ARG, "A, B and D must be non-NULL and 16-byte aligned");
  cudaError_t e = dfv::launch_mma_selftest(A, B, D, dtype == DFV_BF16 ? 1 : 0, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "MMA self-test launch");
  return DFV_OK;
}

int dfv_selftest_tcgen05(const void *A, const void *B, int N, int K, float *D, int32_t *status, void *stream) {
  if (N < 16 || N > 256 || N % 16 || (K != 64 && K != 128))
    return fail(DFV_ERR_UNSUPPORTED, "tcgen05 self-test takes N = 16..256 (multiple of 16) and K = 64 or 128");
  if (!A || !B || !D || !status || !aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
    return fail(DFV_ERR_INVALID_ARG, "A, B, D and status must be non-NULL, A, B and D 16-byte aligned");
  cudaError_t e = dfv::launch_tc05_selftest(A, B, N, K, D, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 self-test launch");
  return DFV_OK;
}

int dfv_read_device_error(const void *ws, uint32_t *err_host, void *stream) {
  if (!ws || !err_host) return fail(DFV_ERR_INVALID_ARG, "ws and err_host must not be NULL");
  if (!aligned(ws, 256)) return fail(DFV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaError_t e = cudaMemcpyAsync(err_host, (const char *)ws + 256, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "device->host copy of the error word");
  return DFV_OK;
}

size_t dfv_accept_workspace_size(int k_max, int V) {
  if (k_max < 0 || k_max > DFV_MAX_BLOCK || V < 1) return 0;
  return align256(sizeof(unsigned)) + align256((size_t)(k_max + 1) * 304 * 8);
}

int dfv_accept_greedy(const void *logits, int dtype, int k, int V, const int32_t *draft, int32_t *tau,
                      int32_t *committed, void *ws, size_t ws_bytes, void *stream) {
  if (k < 0 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 0..%d", k, DFV_MAX_BLOCK);
  if (V < 1) return fail(DFV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (dtype != DFV_BF16 && dtype != DFV_F32) return fail(DFV_ERR_UNSUPPORTED, "logits dtype %d", dtype);
  if (!logits || !aligned(logits, 16) || !tau || (k > 0 && !draft))
    return fail(DFV_ERR_INVALID_ARG, "logits/tau/draft NULL or logits not 16-byte aligned");
  if (!ws || !aligned(ws, 256)) return fail(DFV_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < dfv_accept_workspace_size(k, V))
    return fail(DFV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, dfv_accept_workspace_size(k, V));
  dfv::AcceptParams p = {};
  p.logits = logits;
  p.draft = draft;
  p.tau = tau;
  p.committed = committed;
  p.k = k;
  p.V = V;
  p.dtype = dtype;
  int chunks = (304 + k) / (k + 1);  // about two CTAs per SM in total
  const int maxc = (V + 1023) / 1024;
  if (chunks > maxc) chunks = maxc;
  if (chunks < 1) chunks = 1;
  p.chunks = chunks;
  p.cnt = (unsigned *)ws;
  p.partial = (unsigned long long *)((char *)ws + align256(sizeof(unsigned)));
  cudaError_t e = dfv::launch_accept(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  return DFV_OK;
}

int dfv_accept_greedy_noalloc(const void *logits, int dtype, int k, int V, const int32_t *draft, int32_t *tau,
                              int32_t *committed, void *stream) {
  if (k < 0 || k > DFV_MAX_BLOCK) return fail(DFV_ERR_INVALID_ARG, "k=%d outside 0..%d", k, DFV_MAX_BLOCK);
  if (V < 1) return fail(DFV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (dtype != DFV_BF16 && dtype != DFV_F32) return fail(DFV_ERR_UNSUPPORTED, "logits dtype %d", dtype);
  if (!logits || !aligned(logits, 16) || !tau || (k > 0 && !draft))
    return fail(DFV_ERR_INVALID_ARG, "logits/tau/draft NULL or logits not 16-byte aligned");
  int chunks = (304 + k) / (k + 1);
  const int maxc = (V + 1023) / 1024;
  if (chunks > maxc) chunks = maxc;
  if (chunks < 1) chunks = 1;
  if (chunks > dfv::accept_noalloc_max_chunks())
    return fail(DFV_ERR_UNSUPPORTED, "%d vocabulary slices exceed the fixed scratch (%d)", chunks,
                dfv::accept_noalloc_max_chunks());
  void *scratch = nullptr;
  cudaError_t e = dfv::accept_noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "fixed scratch lookup (cudaGetSymbolAddress)");
  cudaStream_t s = (cudaStream_t)stream;
  // the ticket must start at zero: clear it in stream order (no allocation)
  e = cudaMemsetAsync(scratch, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the fixed scratch ticket");
  dfv::AcceptParams p = {};
  p.logits = logits;
  p.draft = draft;
  p.tau = tau;
  p.committed = committed;
  p.k = k;
  p.V = V;
  p.dtype = dtype;
  p.chunks = chunks;
  p.cnt = (unsigned *)scratch;
  p.partial = (unsigned long long *)scratch + 32;
  e = dfv::launch_accept(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  return DFV_OK;
}

}  // extern "C"
