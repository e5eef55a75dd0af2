/*
 * oracle.h -- plain CPU oracle for the MoE block-verify step of DFlash-style
 * speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference leg may load this library.  The product path (the
 * CUDA library and its Python binding) never calls it, links it or shares code
 * with it.
 *
 * Every function computes in IEEE double precision from inputs decoded exactly
 * (bf16 and fp32 widen exactly to double; mxfp4 values are exact binary
 * numbers).  Where a floating-point value decides an integer (the top-K
 * selection), the decision is taken on the value rounded to fp32, which is the
 * precision the GPU kernels decide in.
 *
 * Sources (page titles and sections of the method's write-ups):
 *   [P1] "Speculating on a Strix Halo", sections "Speculative decoding",
 *        "What the pieces cost" (including its always-on shared expert),
 *        "The verify's own cost", reference 1 (model card: 256 experts, 8
 *        routed plus 1 shared activated).
 *   [P2] "Speculating on a Strix Halo (part 2)", sections "The verification
 *        cog", "Why drafter performance doesn't really matter", "Two bugs
 *        upstream".
 *   [P3] the MI355X / vLLM write-up at allbreaknews.com/?p=4397, sections
 *        "Why Quantize the Target Model on Top?" and "Results: Quantizing
 *        the Target Model" (mxfp4 target weights).
 *
 * Array conventions: row-major, contiguous.  dtype codes below.  bf16 arrays
 * are passed as their raw 16-bit patterns.  mxfp4 matrices are passed as
 * packed nibbles [rows][cols/2] (low nibble = even column) plus one e8m0 scale
 * byte per 32 consecutive elements of a row, [rows][cols/32].  q8 matrices are
 * passed as int8 codes [rows][cols] plus one IEEE binary16 scale per 32
 * consecutive elements of a row, [rows][cols/32] (through the `scales`
 * pointer); element value = code * scale.
 */
#ifndef DFV_ORACLE_H
#define DFV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_MXFP4 = 2, ORC_Q8 = 3, ORC_F16 = 4 /* IEEE binary16 */ };

typedef struct {
  int d, n_experts, top_k, d_ff, norm_topk;
  int w_dtype, r_dtype;           /* expert / router weight dtypes */
  const void *w_router;           /* [E][d] */
  const void *w_gate, *w_up;      /* [E][d_ff][d]  (mxfp4: bytes [E][d_ff][d/2]) */
  const void *w_down;             /* [E][d][d_ff]  (mxfp4: bytes [E][d][d_ff/2]) */
  const uint8_t *s_gate, *s_up, *s_down; /* e8m0 scales (mxfp4 only) */
  int n_shared;  /* 0 or 1: one always-on shared expert, stored as expert E of
                    w_gate / w_up / w_down (and their scales); the router has
                    E rows only */
} orc_layer;

/* scalar helpers */
double   orc_bf16_to_double(uint16_t bits);
uint16_t orc_double_to_bf16(double v);          /* round to nearest, ties to even */
double   orc_e2m1_value(int code);              /* 4-bit code -> value */
double   orc_e8m0_value(int e);                 /* 2^(e-127) */
double   orc_fp16_to_double(uint16_t bits);     /* IEEE binary16, exact */
double   orc_silu(double z);

/* decode rows [r0, r0+nrows) of a (possibly mxfp4) matrix with `cols` columns */
int orc_decode_rows(int dtype, const void *data, const uint8_t *scales,
                    int r0, int nrows, int cols, double *out);

/* router: logits (rounded to fp32), top-K indices, routing weights */
/* D[M][N] = A[M][L] . B[L][N] in double (operands F32, BF16 or F16). */
int orc_matmul(int dtype, const void *A, const void *B, int M, int L, int N,
               double *D);

int orc_route(const orc_layer *L, const void *x, int x_dtype, int k,
              float *logits, int32_t *topk_idx, double *topk_w);

/* union of woken experts, offsets and (expert, token)-sorted gather list */
int orc_woken(int k, int K, int E, const int32_t *topk_idx,
              int32_t *woken, int32_t *n_woken, int32_t *offsets,
              int32_t *gather);

/* one expert on one token row: y = W_down (silu(W_gate x) * (W_up x)) */
int orc_expert_ffn(const orc_layer *L, int e, const double *x, double *y);

/* MoE output of one layer (routed experts, plus the shared expert when
 * n_shared = 1), out[k][d] in double */
int orc_moe_forward(const orc_layer *L, const void *x, int x_dtype, int k,
                    double *out, int nthreads);

/* RMSNorm with unit gain */
int orc_rmsnorm(const void *x, int x_dtype, int k, int d, double eps,
                double *out);

/* residual stack of MoE layers, bf16 residual stream */
int orc_stack_forward(const orc_layer *layers, int n_layers,
                      const uint16_t *x_in, int k, double eps,
                      uint16_t *x_out, int nthreads);

/* greedy acceptance */
int orc_argmax_rows(const void *logits, int dtype, int rows, int V,
                    int32_t *a);
int orc_accept_greedy(const void *logits, int dtype, int k, int V,
                      const int32_t *draft, int32_t *tau,
                      int32_t *committed);

int orc_num_threads_available(void);

#ifdef __cplusplus
}
#endif
#endif
