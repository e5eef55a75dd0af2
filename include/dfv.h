/*
 * dfv.h -- C ABI of the GB300 (sm_103a) MoE block-verify library, libdfv.so.
 *
 * The target model's verify step in DFlash-style speculative decoding over a
 * Mixture-of-Experts model: a block of k drafted positions goes through each
 * MoE layer together, and greedy acceptance turns the target's logits into the
 * committed length tau.
 *
 * Sources (page titles and sections of the method's write-ups):
 *   "Speculating on a Strix Halo", section "Speculative decoding": the target
 *       checks the whole draft in one pass; under greedy decoding it accepts
 *       only tokens it would have produced itself; a cycle commits the accepted
 *       draft prefix plus one token of the target's own (tau).
 *   same page, section "What the pieces cost": each token of the block routes
 *       to its own experts, so the block wakes the union of its rows' experts;
 *       reference 1 (model card): 8 routed experts of 256.
 *   same page, section "The verify's own cost": tokens are sorted by expert
 *       and each projection runs as one grouped launch.
 *   "Speculating on a Strix Halo (part 2)", section "The verification cog":
 *       the verifier is the base model run over the draft; expert weight
 *       streaming is what makes verify cost more than decode.
 *   same page, section "Why drafter performance doesn't really matter": the
 *       n-th drafted token is accepted only if the n-1 before it were.
 *   same page, section "What the pieces cost", and its reference 1: one
 *       always-on shared expert besides the 8 routed ones.
 *   the MI355X / vLLM write-up (allbreaknews.com/?p=4397), sections "Why
 *       Quantize the Target Model on Top?" and "Results: Quantizing the Target
 *       Model": mxfp4 target weights, used natively, never re-materialised.
 *
 * Conventions for every entry point:
 *   - Pointers named in the signatures are DEVICE pointers, owned by the
 *     caller, unless a comment says "host".  Tensors are row-major and
 *     contiguous.  Every pointer must be 16-byte aligned; the workspace
 *     256-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on it and returns; nothing is synchronised and
 *     nothing is allocated.  Arguments are validated on the host before any
 *     launch; on a non-zero status nothing was enqueued (except DFV_ERR_CUDA,
 *     where a launch itself failed).
 *   - Workspaces are caller-owned device memory of at least the size the
 *     matching *_workspace_size() reports.  A workspace must be ZERO-FILLED
 *     before its first use (e.g. cudaMemset); every call leaves it zero-ready
 *     for the next one (the counters that must start at zero live at fixed
 *     offsets, so one workspace serves any k and, for d <= 13312, any layer).
 *     Calls that share a workspace must be ordered (same stream, or
 *     synchronised): concurrent use races.
 *   - Returns DFV_OK (0) or a DFV_ERR_* status; dfv_status_string() names it
 *     and dfv_last_error_detail() gives the last failure's detail text
 *     (thread-local).
 */
#ifndef DFV_H
#define DFV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFV_VERSION 2

enum {
  DFV_OK = 0,
  DFV_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, size out of range  */
  DFV_ERR_UNSUPPORTED = 2,  /* dtype combination or shape not supported   */
  DFV_ERR_WORKSPACE = 3,    /* workspace too small or misaligned          */
  DFV_ERR_CUDA = 4          /* a CUDA launch or copy failed               */
};

/* DFV_Q8: 8-bit expert weights (see dfv_moe_layer).  DFV_F16 (IEEE binary16)
 * appears only in dfv_selftest_mma. */
typedef enum { DFV_F32 = 0, DFV_BF16 = 1, DFV_MXFP4 = 2, DFV_Q8 = 3, DFV_F16 = 4 } dfv_dtype;

/* Device-side error bits a kernel may set in the workspace (see
 * dfv_read_device_error).  Every wait inside a kernel is bounded; a wait that
 * runs out sets one of these bits and the kernel returns early (its outputs
 * are then invalid). */
#define DFV_DEVERR_STAGE_WAIT 0x1u   /* a consumer gave up waiting for a weight tile */
#define DFV_DEVERR_SLOT_WAIT 0x2u    /* the producer gave up waiting for a free stage */
#define DFV_DEVERR_DRAIN_WAIT 0x4u   /* copies still in flight at exit after a timeout */
#define DFV_DEVERR_GRID_WAIT 0x8u    /* a CTA gave up waiting at a grid-wide barrier */
/* Reserved; no kernel sets it.  It once flagged mxfp4 scale bytes outside the
 * range that a scale folded into fp16 codes keeps exact.  Every mxfp4 path
 * (single launch and multi-launch) now multiplies each 32-element block's
 * fp32 partial sum by its scale 2^(s-127), exact for every scale 0..254. */
#define DFV_DEVERR_SCALE_RANGE 0x10u
#define DFV_DEVERR_REDUCE_WAIT 0x20u /* a warp gave up waiting for a free partial-sum buffer */
/* A single-launch kernel found its own routing tables inconsistent (an expert
 * id, offset or pair index out of range, or a pair filed under the wrong
 * expert) and skipped the layer's expert work rather than index with them. */
#define DFV_DEVERR_ROUTING 0x40u

/* Limits of this implementation. */
#define DFV_MAX_BLOCK 16      /* k: positions in one verify block          */
#define DFV_MAX_EXPERTS 256   /* E                                          */
#define DFV_MAX_TOPK 8        /* K                                          */
#define DFV_MAX_BATCH_ROWS 512 /* n_blocks * k in one batched verify call     */

/*
 * One MoE layer.  All weights are caller-owned device memory.
 *   w_router  [E, d]            router weights, r_dtype (F32 or BF16)
 *   w_gate    [E, d_ff, d]      gate projection of every expert
 *   w_up      [E, d_ff, d]      up projection
 *   w_down    [E, d, d_ff]      down projection
 * For w_dtype = DFV_MXFP4 the three expert matrices hold packed E2M1 codes,
 * two per byte, low nibble = even column ([E, d_ff, d/2], [E, d, d_ff/2]
 * bytes), and s_gate/s_up/s_down hold one E8M0 scale byte per 32 consecutive
 * elements of a row ([E, d_ff, d/32], [E, d_ff, d/32], [E, d, d_ff/32]);
 * element value = e2m1(code) * 2^(scale - 127).  Scale 255 (NaN) is not
 * supported.
 * For w_dtype = DFV_Q8 (8-bit weights; the pages run the target "at Q8" and
 * fix no format, read here as llama.cpp's Q8_0 block: 32 int8 codes of a row
 * share one IEEE binary16 scale) the expert matrices hold int8 codes ([E,
 * d_ff, d], [E, d, d_ff]) and s_gate/s_up/s_down one binary16 scale per 32
 * consecutive elements of a row, as uint16 patterns ([E, d_ff, d/32], ...);
 * element value = code * scale.  Scales must be finite.
 * For F32/BF16 weights the scale pointers are ignored.
 * norm_topk: 1 renormalises the K selected routing weights to sum 1
 * (w_s = p_s / sum p), 0 keeps the softmax probabilities p_s.
 * n_shared: 0, or 1 for one always-on shared expert ("What the pieces cost":
 * the routed experts plus an always-on shared one).  It has the routed
 * experts' form and size and is stored as expert index E of w_gate / w_up /
 * w_down (and of s_gate / s_up / s_down), so those arrays then hold E + 1
 * experts; w_router stays [E, d].  Every row of the block goes through it and
 * its output is added with weight 1 after the routed sum.  (The pages give it
 * no gate; none is applied.)
 * Supported combinations (w_dtype, r_dtype, activations):
 *   (BF16, BF16, BF16), (MXFP4, BF16, BF16), (Q8, BF16, BF16), (F32, F32, F32).
 * Shapes: 1 <= K <= min(E, 8), E <= 256, d % 32 == 0, d_ff % 32 == 0
 * (MXFP4: d % 64 == 0 and d_ff % 64 == 0).  Block-scaled layers run in one
 * launch when d % 512 == 0 (Q8: d % 256 == 0), d <= 2048, 64 <= d_ff <= 512
 * and d_ff % 128 == 0 (Q8: d_ff % 64 == 0, and d_ff % 256 == 0 above 256);
 * other MXFP4 shapes take the multi-kernel path, other Q8 shapes are
 * DFV_ERR_UNSUPPORTED.
 */
typedef struct dfv_moe_layer {
  int d, n_experts, top_k, d_ff, norm_topk;
  int w_dtype; /* dfv_dtype of the expert weights */
  int r_dtype; /* dfv_dtype of the router weights */
  const void *w_router;
  const void *w_gate, *w_up, *w_down;
  const uint8_t *s_gate, *s_up, *s_down;
  int n_shared; /* 0 or 1 */
} dfv_moe_layer;

/* Bytes of workspace dfv_route_topk / dfv_moe_block_forward /
 * dfv_moe_stack_forward need for blocks of up to k_max positions
 * (0 on invalid arguments).  A layer with a shared expert needs more. */
size_t dfv_moe_workspace_size(const dfv_moe_layer *layer, int k_max);

/*
 * Router of one layer for a block of k positions ("What the pieces cost":
 * each token routes to its own experts; the block wakes their union).
 *   hidden    [k, d] activations (act = BF16 or F32, matching the layer)
 * Outputs (device, caller-owned; any may be NULL except n_woken):
 *   topk_idx  [k, K] int32   experts of each row, by descending router logit,
 *                            equal logits ordered by lower expert index
 *   topk_w    [k, K] fp32    routing weights (softmax over all E logits,
 *                            renormalised over the K when norm_topk)
 *   woken     [min(E, k*K)]  int32, ascending ids of the woken experts
 *   n_woken   [1]  int32     W, the number of woken experts
 *   offsets   [W + 1] int32  exclusive prefix sum of per-expert pair counts
 *   gather    [k*K] int32    flat pair ids t*K+s ordered by (expert, t)
 * Logits are fp32 dot products of the given operands; selection compares
 * those fp32 values exactly.
 */
int dfv_route_topk(const dfv_moe_layer *layer, const void *hidden, int act, int k,
                   int32_t *topk_idx, float *topk_w, int32_t *woken, int32_t *n_woken,
                   int32_t *offsets, int32_t *gather, void *ws, size_t ws_bytes, void *stream);

/*
 * Enqueue a copy of the workspace's device error word (DFV_DEVERR_* bits, 0 =
 * no error) to host memory `err_host` on `stream`; read it after the stream
 * has synchronised.  The bits are sticky: after a non-zero word the outputs of
 * the calls since the workspace was zero-filled are invalid, and the
 * workspace must be zero-filled again before reuse.  (No counterpart on the
 * method's pages: the bounded waits of the TMA-staged kernels report here.)
 */
int dfv_read_device_error(const void *ws, uint32_t *err_host, void *stream);

/*
 * Expert output of one MoE layer for a block of k positions: router,
 * top-K, woken-expert union and per-expert token gather, SwiGLU expert FFN
 *   y = W_down (silu(W_gate x) * (W_up x)),  silu(z) = z / (1 + e^-z),
 * and the routing-weighted combine out[t] = sum_s w[t,s] y_{idx[t,s]}(x[t]),
 * summed in slot order, + y_E(x[t]) when n_shared = 1 ("What the pieces
 * cost"; "The verify's own cost").  The residual is not included.  The
 * shared expert runs as one more woken expert that every row selects.
 *   hidden  [k, d] act   input rows
 *   out     [k, d] act   output (bf16 or fp32, same dtype as hidden)
 *   opt_topk_idx [k, K] int32 and opt_n_woken [1] int32: optional copies of
 *           the routing decision (NULL to skip); n_woken counts the routed
 *           experts only.
 * Accumulation is fp32.  Each weight byte of a woken expert is read from HBM
 * once per call; experts no row selected are not read.
 */
int dfv_moe_block_forward(const dfv_moe_layer *layer, const void *hidden, int act, int k,
                          void *out, int32_t *opt_topk_idx, int32_t *opt_n_woken,
                          void *ws, size_t ws_bytes, void *stream);

/*
 * Same as dfv_moe_block_forward, but `hidden_host` and `out_host` are HOST
 * buffers (pinned memory gives asynchronous copies).  The call enqueues the
 * host->device copy of hidden into the workspace, the layer, and the
 * device->host copy of out; the caller synchronises the stream before reading
 * out_host.  The workspace must be sized with dfv_moe_workspace_size.
 */
int dfv_moe_block_forward_host(const dfv_moe_layer *layer, const void *hidden_host, int act, int k,
                               void *out_host, void *ws, size_t ws_bytes, void *stream);

/*
 * Pre-norm residual stack of MoE layers over a bf16 residual stream, in place:
 *   n_l     = bf16(x_l / sqrt(mean(x_l^2) + eps))      (RMSNorm, unit gain)
 *   x_{l+1} = bf16(x_l + MoE_l(n_l))                    (one rounding)
 *   layers  host array of n_layers layer descriptors (BF16, MXFP4 or Q8 experts,
 *           BF16 router), all with the same d
 *   x       [k, d] bf16 device buffer, input and output
 *   opt_n_woken  NULL, or an int32 device array [n_layers]: per layer, the
 *           number of distinct routed experts the block woke
 * Layers are applied in order; each one's routing depends on the previous
 * one's output ("Speculating on a Strix Halo (part 2)", section "The
 * verification cog": every layer pays its own fixed cost, which is what the
 * decode step of one token feels).  When every layer has bf16 experts and
 * router and the same shape (d, d_ff, experts, top-k, shared expert, weight
 * renormalisation), and the single-launch kernel fits the shape, the layers
 * can run as ONE persistent cooperative launch per 48 layers: grid barriers
 * separate the layers, the next layer's router rows are fetched towards L2
 * while the current one drains, and no launch or set-up is paid in between
 * (see dfv_set_stack_launch).  Otherwise one launch (or one multi-kernel
 * sequence) per layer.  Both give the same bits.  The workspace is sized for
 * the largest layer with dfv_moe_workspace_size; one error word covers the
 * whole call.
 */
int dfv_moe_stack_forward(const dfv_moe_layer *layers, int n_layers, void *x, int k, float eps,
                          int32_t *opt_n_woken, void *ws, size_t ws_bytes, void *stream);

/* Bytes of workspace dfv_moe_batch_forward needs for up to n_rows_max rows
 * (n_blocks * k) of a layer (0 on invalid arguments). */
size_t dfv_moe_batch_workspace_size(const dfv_moe_layer *layer, int n_rows_max);

/*
 * Batched verify: n_blocks verify blocks of k positions each (T = n_blocks * k
 * <= 512 rows, e.g. 32 concurrent requests with 16-token blocks; the MI355X /
 * vLLM write-up, section "Results: Throughput and Speedup", serves up to 32)
 * through one MoE layer, every row routed on its own exactly as in
 * dfv_moe_block_forward:
 *   out[t] = sum_s w[t,s] y_{idx[t,s]}(x[t])  (+ y_E(x[t]) with a shared expert)
 * Rows of different blocks share nothing but the weights: each woken expert's
 * weights are streamed once for all rows of all blocks that route to it.
 *   hidden [T, d] bf16 rows, block b in rows [b k, (b+1) k)
 *   out    [T, d] bf16
 *   opt_topk_idx [T, K] int32, opt_n_woken [1] int32 (routed experts woken
 *          by the whole batch): optional copies of the routing (NULL to skip)
 * Supported: bf16 experts and router, d % 128 == 0, d_ff % 128 == 0,
 * d <= 8192.  Row t's routing equals dfv_moe_block_forward's on the block
 * holding t (the same fp32 logits); the expert contractions run on the
 * fifth-generation tensor cores, fp32 accumulation, h rounded to bf16.
 * The workspace needs no zero-filling: every call rewrites what it reads.
 */
int dfv_moe_batch_forward(const dfv_moe_layer *layer, const void *hidden, int n_blocks, int k, void *out,
                          int32_t *opt_topk_idx, int32_t *opt_n_woken, void *ws, size_t ws_bytes, void *stream);

/* Bytes of workspace dfv_accept_greedy needs for up to k_max drafted tokens
 * over a vocabulary of V (0 on invalid arguments). */
size_t dfv_accept_workspace_size(int k_max, int V);

/*
 * Greedy acceptance ("Speculative decoding": the target accepts only tokens it
 * would have produced itself and commits the accepted prefix plus one token of
 * its own; part 2, "Why drafter performance doesn't really matter": the n-th
 * draft is accepted only if the n-1 before it were).
 *   logits    [k+1, V] (BF16 or F32) target logits at the k+1 positions
 *   draft     [k] int32 drafted tokens, 0 <= k <= 16
 *   a[i]      = argmax_v logits[i, v], equal values to the lowest v
 *               (+0 and -0 compare equal; logits must not be NaN)
 *   n         = largest j <= k with draft[i] == a[i] for all i < j
 *   tau       [1] int32  = n + 1
 *   committed [k+1] int32 or NULL: a[0..n], then -1
 */
int dfv_accept_greedy(const void *logits, int dtype, int k, int V, const int32_t *draft,
                      int32_t *tau, int32_t *committed, void *ws, size_t ws_bytes, void *stream);

/*
 * Profiling hook (no counterpart on the method's pages; used to time each
 * kernel of the layer with CUDA events).  With a non-NULL array of 4
 * cudaEvent_t handles, every later layer call made from this host thread
 * records events[0] before the router launch, events[1] after it, events[2]
 * after the gate/up launch and events[3] after the down/combine launch, on the
 * call's stream.  NULL turns it off.  The events are caller-owned; recording
 * them between launches keeps the launches in stream order but removes the
 * overlap of one kernel's start with the previous kernel's tail.
 */
int dfv_profile_set_events(void *const *events, int n_events);

/*
 * Kernel path for later layer calls from this host thread (no counterpart on
 * the method's pages).  1 (default): bf16 layers whose shape fits run as one
 * cooperative persistent launch per layer (router, routing, gate/up, down and
 * combine separated by grid-wide barriers); the others, and 0, use the
 * multi-kernel path (router launch, then gate/up and down/combine launches).
 * Both compute the same function.  With the fused path the profiling events
 * 1-3 are recorded together after the single launch.
 */
int dfv_set_path(int path);

/*
 * How dfv_moe_stack_forward launches a stack whose layers allow the persistent
 * kernel, for later calls from this host thread (no counterpart on the
 * method's pages):
 *   0  one launch per layer (chained programmatically);
 *   1  (default) one persistent launch per 48 layers when k <= 8 and the
 *      stream is not capturing a CUDA graph, else one launch per layer.  Measured
 *      on GB300 (40 Qwen3-A3B-like layers): eager calls at k = 1 take 28.8 us
 *      per layer persistent against 30.8 us per launch, but inside a graph the
 *      chained launches take 27.7 us against 28.8 us; at k = 16 the persistent
 *      kernel's down loop spills registers (173 against 133-137 us);
 *   2  one persistent launch per 48 layers for every k.
 * The result is the same bit for bit.  Returns DFV_ERR_INVALID_ARG for a mode
 * outside 0..2.
 */
int dfv_set_stack_launch(int mode);

/* Path the last layer call from this host thread took: 1 fused, 0
 * multi-kernel, 2 batched verify (dfv_moe_batch_forward), 3 persistent stack
 * launch (dfv_moe_stack_forward), -1 none yet.  With profiling events set, a
 * persistent stack call records events[0] before and events[1..3] after each
 * of its launches.
 * With profiling events set, a batched call records events[0] before its
 * routing launches, events[1] after the routing and the token gather,
 * events[2] after the gate/up contraction and events[3] after the down
 * contraction and the combine. */
int dfv_last_layer_path(void);

/*
 * How the single-launch bf16 kernel fetches its gate/up stages, for later
 * layer calls from this host thread (no counterpart on the method's pages):
 * the highest mode allowed: 3 (default) one 3-D tensor-map copy per weight
 * matrix and stage in 128-byte segments with the 128-byte swizzle (d and the
 * stage width multiples of 64), 2 one 3-D tensor-map copy per matrix and stage
 * in 256-column blocks, 1 one 2-D tensor-map copy per 256 columns, 0 one 1-D
 * bulk copy per weight row.  A mode the driver or the shape does not allow
 * falls back to the next lower one.  All modes compute the same result bit for
 * bit.  Mode 0 also makes the multi-launch bf16 path use one bulk copy per
 * weight row for its gate/up stages (its swizzled copies otherwise).
 * Returns DFV_ERR_INVALID_ARG for a mode outside 0..3.
 */
int dfv_set_staging(int max_mode);

/* Staging mode the last single-launch bf16 layer call from this host thread
 * used (see dfv_set_staging), -1 none yet. */
int dfv_last_staging(void);

/* Why the fused path could not be set up on this device (empty if it could,
 * or if it was never tried). */
const char *dfv_fused_unavailable_reason(void);

/*
 * Allocation-free greedy acceptance.  The method's pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory (a
 * runtime with a fixed memory budget, or plain C host code with no allocator
 * of its own to create the workspace dfv_accept_greedy needs).  It computes
 * exactly what dfv_accept_greedy computes, with the same arguments minus the
 * workspace; logits, draft, tau and committed are still the caller's device
 * buffers.
 * Its scratch is a fixed device array inside libdfv.so (about 41 KB, enough
 * for every k <= 16 and any V) that each GPU holds until the process exits.
 * The first call in a CUDA context (per device, and again after
 * cudaDeviceReset) looks the array's device address up (cudaGetSymbolAddress)
 * and keeps it for that context, so make that first call before any stream
 * capture.
 * Each call clears the array's ticket with cudaMemsetAsync on `stream` and
 * allocates nothing.  All calls share the array: calls whose kernels overlap
 * on the GPU race; order them (one stream, or synchronise).
 * Returns DFV_ERR_UNSUPPORTED if a launch would need more vocabulary slices
 * than the array holds (cannot happen within the documented limits).
 */
int dfv_accept_greedy_noalloc(const void *logits, int dtype, int k, int V, const int32_t *draft,
                              int32_t *tau, int32_t *committed, void *stream);

/*
 * Self-test of the device-side bounded waits (no counterpart on the method's
 * pages).  One launch of one thread waits on an mbarrier phase that nothing
 * completes, then on a grid barrier that its single CTA can never fill.  Both
 * are the waits the single-launch kernels use, with their limit (2 s): each
 * gives up, sets its bit in the workspace error word (DFV_DEVERR_STAGE_WAIT,
 * DFV_DEVERR_GRID_WAIT) and returns.  The call takes about 4 s of GPU time;
 * no copy is in flight when a wait gives up, and the context stays usable.
 * Read the word with dfv_read_device_error, then zero-fill the workspace
 * before other calls use it.
 *   ws  a zero-filled workspace of any dfv_moe_workspace_size() (the
 *       counters sit in its first 8 KB).
 */
int dfv_selftest_bounded_waits(void *ws, size_t ws_bytes, void *stream);

/*
 * Self-test of the tensor-core fragment path the expert kernels use (its
 * instance comes from "Speculating on a Strix Halo (part 2)", section "Two
 * bugs upstream": a multiply-add with an exact result must return it whatever
 * the sign of its zero operands).  One warp computes
 *   D[i][j] = sum_l A[i][l] * B[l][j]      (16 x 16 x 16, fp32 accumulate)
 * with the MMA helper and operand mapping of the bf16 kernels (dtype
 * DFV_BF16) or of the mxfp4 kernels (DFV_F16: binary16 operands).
 *   A, B  [16][16] 16-bit elements (device), row-major
 *   D     [16][16] fp32 (device)
 * Returns DFV_ERR_UNSUPPORTED for another dtype.
 */
int dfv_selftest_mma(int dtype, const void *A, const void *B, float *D, void *stream);

/*
 * Self-test of the fifth-generation tensor-core path the batched kernels use
 * (no counterpart on the method's pages): one CTA computes
 *   D[i][j] = sum_l A[i][l] * B[j][l]     (128 x N x K, bf16 in, fp32 out)
 * with the operands in shared memory (128-byte swizzled, K-major), tcgen05
 * MMAs into tensor memory and tcgen05 loads back.
 *   A [128][K], B [N][K] bf16 (device), D [128][N] fp32 (device)
 *   N = 16..256, a multiple of 16; K = 64 or 128
 *   status [1] int32 (device, zeroed by the caller): 1 if the bounded wait
 *   for the MMAs gave up (D is then not written).
 */
int dfv_selftest_tcgen05(const void *A, const void *B, int N, int K, float *D, int32_t *status, void *stream);

const char *dfv_status_string(int status);
const char *dfv_last_error_detail(void);
int dfv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DFV_H */
