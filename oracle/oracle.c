/*
 * oracle.c -- plain CPU oracle for the MoE block-verify step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Shares no code with the CUDA
 * library.  Loops are written in the order the definitions state them; the
 * only parallelism (optional OpenMP over independent (token, slot) pairs in
 * orc_moe_forward) does not change any result, because every pair is computed
 * by the same sequential code and the combine runs afterwards in slot order.
 *
 * Where the method's pages leave a step open, the reading taken is stated at
 * the function.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* scalar formats                                                      */
/* ------------------------------------------------------------------ */

double orc_bf16_to_double(uint16_t bits) {
  /* bf16 is the upper half of an IEEE binary32 pattern: widening is exact */
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t orc_double_to_bf16(double v) {
  /* Round to the nearest bf16 value, ties to even (8 significant bits,
   * exponent range of binary32, subnormal quantum 2^-133). */
  if (isnan(v)) return 0x7fc0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);            /* a in [2^(e-1), 2^e) */
  int q = e - 8;                 /* weight of the last kept bit */
  if (q < -133) q = -133;
  double r = nearbyint(ldexp(a, -q)); /* default mode: ties to even */
  double rv = ldexp(r, q);
  float f = (float)rv;           /* exact, or +inf on overflow */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

/* OCP microscaling element format E2M1: 1 sign bit, 2 exponent bits (bias 1),
 * 1 mantissa bit.  The eight magnitudes are listed once here. */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code) {
  double m = kE2M1Magnitude[code & 7];
  return (code & 8) ? -m : m;
}

double orc_e8m0_value(int e) {
  /* E8M0 shared scale: 2^(e-127); the all-ones pattern encodes NaN. */
  if (e == 255) return NAN;
  return ldexp(1.0, e - 127);
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds zero and the subnormals (fraction * 2^-24), exponent
 * 31 infinity and NaN.  Every value widens exactly to double. */
double orc_fp16_to_double(uint16_t bits) {
  int sign = bits >> 15, e = (bits >> 10) & 31, f = bits & 1023;
  double m;
  if (e == 0) m = ldexp((double)f, -24);
  else if (e == 31) m = f ? NAN : INFINITY;
  else m = ldexp((double)(1024 + f), e - 25);
  return sign ? -m : m;
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

int orc_decode_rows(int dtype, const void *data, const uint8_t *scales,
                    int r0, int nrows, int cols, double *out) {
  if (!data || !out || nrows < 0 || cols <= 0) return -1;
  for (int r = 0; r < nrows; ++r) {
    size_t row = (size_t)(r0 + r);
    for (int c = 0; c < cols; ++c) {
      double v;
      if (dtype == ORC_F32) {
        v = (double)((const float *)data)[row * cols + c];
      } else if (dtype == ORC_BF16) {
        v = orc_bf16_to_double(((const uint16_t *)data)[row * cols + c]);
      } else if (dtype == ORC_MXFP4) {
        if (!scales || cols % 32) return -1;
        uint8_t byte = ((const uint8_t *)data)[row * (cols / 2) + c / 2];
        int code = (c & 1) ? (byte >> 4) : (byte & 15);
        int s = scales[row * (cols / 32) + c / 32];
        v = orc_e2m1_value(code) * orc_e8m0_value(s);
      } else if (dtype == ORC_Q8) {
        /* 8-bit weights, read as llama.cpp's Q8_0 block: 32 int8 codes of a
         * row share one binary16 scale (codes and scales kept in two arrays,
         * like the mxfp4 ones) */
        if (!scales || cols % 32) return -1;
        int code = ((const int8_t *)data)[row * cols + c];
        uint16_t s = ((const uint16_t *)scales)[row * (cols / 32) + c / 32];
        v = (double)code * orc_fp16_to_double(s);
      } else if (dtype == ORC_F16) {
        v = orc_fp16_to_double(((const uint16_t *)data)[row * cols + c]);
      } else {
        return -1;
      }
      out[(size_t)r * cols + c] = v;
    }
  }
  return 0;
}

static int act_ok(int dt) { return dt == ORC_F32 || dt == ORC_BF16; }

/*
 * Plain matrix product of decoded operands, the contraction inside every
 * expert projection:  D[i][j] = sum over l of A[i][l] * B[l][j]  for A [M][L]
 * and B [L][N] of one element format (F32, BF16 or F16), summed in double in
 * the order l = 0, 1, ... .  "Speculating on a Strix Halo (part 2)", section
 * "Two bugs upstream", prints a 16x16 instance whose exact result a correct
 * multiply-add must return whatever the sign of its zero operands.
 */
int orc_matmul(int dtype, const void *A, const void *B, int M, int L, int N,
               double *D) {
  if (M < 1 || L < 1 || N < 1 ||
      !(dtype == ORC_F32 || dtype == ORC_BF16 || dtype == ORC_F16))
    return -1;
  double *a = malloc(sizeof(double) * (size_t)M * L);
  double *b = malloc(sizeof(double) * (size_t)L * N);
  if (!a || !b) return -2;
  orc_decode_rows(dtype, A, NULL, 0, M, L, a);
  orc_decode_rows(dtype, B, NULL, 0, L, N, b);
  for (int i = 0; i < M; ++i)
    for (int j = 0; j < N; ++j) {
      double acc = 0.0;
      for (int l = 0; l < L; ++l) acc += a[(size_t)i * L + l] * b[(size_t)l * N + j];
      D[(size_t)i * N + j] = acc;
    }
  free(a);
  free(b);
  return 0;
}

/* ------------------------------------------------------------------ */
/* router                                                              */
/* ------------------------------------------------------------------ */

/*
 * Per-token routing ([P1] "What the pieces cost": each token routes to its own
 * experts; reference 1: 8 routed of 256).
 *   logits[t][e] = sum_j x[t][j] * Wr[e][j]           (double, then fp32)
 *   top-K: the K largest logits, ordered by (logit desc, index asc)
 *   p = softmax over all E logits
 *   w_s = p[idx_s] / sum_s' p[idx_s']   when norm_topk, else p[idx_s]
 * Reading: the selection is taken on logits, not on rounded probabilities;
 * equal logits go to the lower expert index.
 */
int orc_route(const orc_layer *L, const void *x, int x_dtype, int k,
              float *logits, int32_t *topk_idx, double *topk_w) {
  const int d = L->d, E = L->n_experts, K = L->top_k;
  if (k < 1 || d < 1 || E < 1 || K < 1 || K > E || !act_ok(x_dtype) ||
      !act_ok(L->r_dtype))
    return -1;
  double *xr = malloc(sizeof(double) * d);
  double *wr = malloc(sizeof(double) * d);
  double *z = malloc(sizeof(double) * E);
  char *chosen = malloc(E);
  if (!xr || !wr || !z || !chosen) return -2;

  for (int t = 0; t < k; ++t) {
    orc_decode_rows(x_dtype, x, NULL, t, 1, d, xr);
    for (int e = 0; e < E; ++e) {
      orc_decode_rows(L->r_dtype, L->w_router, NULL, e, 1, d, wr);
      double acc = 0.0;
      for (int j = 0; j < d; ++j) acc += xr[j] * wr[j];
      logits[(size_t)t * E + e] = (float)acc;
    }
    const float *lg = logits + (size_t)t * E;

    memset(chosen, 0, E);
    for (int s = 0; s < K; ++s) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (chosen[e]) continue;
        if (best < 0 || lg[e] > lg[best]) best = e; /* strict: lowest index wins ties */
      }
      chosen[best] = 1;
      topk_idx[t * K + s] = best;
    }

    double m = lg[0];
    for (int e = 1; e < E; ++e)
      if (lg[e] > m) m = lg[e];
    double S = 0.0;
    for (int e = 0; e < E; ++e) {
      z[e] = exp((double)lg[e] - m);
      S += z[e];
    }
    double sel = 0.0;
    for (int s = 0; s < K; ++s) sel += z[topk_idx[t * K + s]] / S;
    for (int s = 0; s < K; ++s) {
      double p = z[topk_idx[t * K + s]] / S;
      topk_w[t * K + s] = L->norm_topk ? p / sel : p;
    }
  }
  free(xr);
  free(wr);
  free(z);
  free(chosen);
  return 0;
}

/* ------------------------------------------------------------------ */
/* woken-expert union and token gather                                 */
/* ------------------------------------------------------------------ */

/*
 * The block wakes the union of its rows' experts ([P1] "What the pieces
 * cost"; [P2] "The verification cog").  Tokens are sorted by expert before the
 * grouped launch ([P1] "The verify's own cost").
 *   woken   : ascending expert ids with at least one routed (token, slot)
 *   offsets : exclusive prefix sum of per-expert counts over `woken`,
 *             offsets[W] = k*K
 *   gather  : the flat pair ids t*K + s, ordered by (expert asc, t asc)
 * Returns W, or a negative value on bad arguments.
 */
int orc_woken(int k, int K, int E, const int32_t *topk_idx, int32_t *woken,
              int32_t *n_woken, int32_t *offsets, int32_t *gather) {
  if (k < 1 || K < 1 || E < 1) return -1;
  int *count = calloc(E, sizeof(int));
  if (!count) return -2;
  for (int p = 0; p < k * K; ++p) {
    int e = topk_idx[p];
    if (e < 0 || e >= E) {
      free(count);
      return -1;
    }
    count[e] += 1;
  }
  int W = 0, off = 0;
  for (int e = 0; e < E; ++e) {
    if (count[e] == 0) continue;
    woken[W] = e;
    offsets[W] = off;
    for (int t = 0; t < k; ++t)
      for (int s = 0; s < K; ++s)
        if (topk_idx[t * K + s] == e) gather[off++] = t * K + s;
    ++W;
  }
  offsets[W] = off;
  *n_woken = W;
  free(count);
  return W;
}

/* ------------------------------------------------------------------ */
/* expert FFN and combine                                              */
/* ------------------------------------------------------------------ */

/*
 * SwiGLU expert: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h, with
 * silu(z) = z / (1 + e^-z).  Weights of expert e are rows [e*rows, (e+1)*rows)
 * of the stacked [E*rows][cols] matrices, decoded exactly to double.
 */
int orc_expert_ffn(const orc_layer *L, int e, const double *x, double *y) {
  const int d = L->d, I = L->d_ff;
  double *row = malloc(sizeof(double) * (d > I ? d : I));
  double *h = malloc(sizeof(double) * I);
  if (!row || !h) return -2;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    orc_decode_rows(L->w_dtype, L->w_gate, L->s_gate, e * I + i, 1, d, row);
    for (int j = 0; j < d; ++j) g += row[j] * x[j];
    orc_decode_rows(L->w_dtype, L->w_up, L->s_up, e * I + i, 1, d, row);
    for (int j = 0; j < d; ++j) u += row[j] * x[j];
    h[i] = orc_silu(g) * u;
  }
  for (int r = 0; r < d; ++r) {
    orc_decode_rows(L->w_dtype, L->w_down, L->s_down, e * d + r, 1, I, row);
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += row[i] * h[i];
    y[r] = acc;
  }
  free(row);
  free(h);
  return 0;
}

/*
 * Output of one MoE layer for a block of k rows:
 *   out[t] = sum over slots s (in slot order) of w[t][s] * FFN_{idx[t][s]}(x[t])
 *            + FFN_E(x[t])                                   (when n_shared = 1)
 * "What the pieces cost" names one always-on shared expert next to the routed
 * ones, and the model card it cites counts "8 routed plus 1 shared" activated
 * experts.  The pages give the shared expert no gate and no weight, so the
 * reading taken is the plainest one: an expert of the same SwiGLU form and
 * size as the routed ones, applied to every row and added with weight 1 after
 * the routed sum.  Its weights are expert index E of the stacked matrices.
 */
int orc_moe_forward(const orc_layer *L, const void *x, int x_dtype, int k,
                    double *out, int nthreads) {
  const int d = L->d, E = L->n_experts, K = L->top_k;
  const int ns = L->n_shared ? 1 : 0;
  if (L->n_shared < 0 || L->n_shared > 1) return -1;
  float *logits = malloc(sizeof(float) * (size_t)k * E);
  int32_t *idx = malloc(sizeof(int32_t) * (size_t)k * K);
  double *w = malloc(sizeof(double) * (size_t)k * K);
  double *xr = malloc(sizeof(double) * (size_t)k * d);
  double *ys = malloc(sizeof(double) * (size_t)k * (K + ns) * d);
  if (!logits || !idx || !w || !xr || !ys) return -2;
  int rc = orc_route(L, x, x_dtype, k, logits, idx, w);
  if (rc) return rc;
  orc_decode_rows(x_dtype, x, NULL, 0, k, d, xr);

  /* pairs t*K+s of the routed experts, then k*K+t of the shared expert */
  int npairs = k * K + k * ns;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int p = 0; p < npairs; ++p) {
    int t = p < k * K ? p / K : p - k * K;
    int e = p < k * K ? idx[p] : E;
    orc_expert_ffn(L, e, xr + (size_t)t * d, ys + (size_t)p * d);
  }
  (void)nthreads;

  for (int t = 0; t < k; ++t) {
    for (int j = 0; j < d; ++j) out[(size_t)t * d + j] = 0.0;
    for (int s = 0; s < K; ++s) {
      const double *y = ys + (size_t)(t * K + s) * d;
      for (int j = 0; j < d; ++j) out[(size_t)t * d + j] += w[t * K + s] * y[j];
    }
    if (ns) {
      const double *y = ys + (size_t)(k * K + t) * d;
      for (int j = 0; j < d; ++j) out[(size_t)t * d + j] += y[j];
    }
  }
  free(logits);
  free(idx);
  free(w);
  free(xr);
  free(ys);
  return 0;
}

/* ------------------------------------------------------------------ */
/* RMSNorm and the residual stack                                      */
/* ------------------------------------------------------------------ */

/* y = x / sqrt(mean(x^2) + eps), unit gain. */
int orc_rmsnorm(const void *x, int x_dtype, int k, int d, double eps,
                double *out) {
  if (!act_ok(x_dtype) || k < 1 || d < 1) return -1;
  double *xr = malloc(sizeof(double) * d);
  if (!xr) return -2;
  for (int t = 0; t < k; ++t) {
    orc_decode_rows(x_dtype, x, NULL, t, 1, d, xr);
    double ss = 0.0;
    for (int j = 0; j < d; ++j) ss += xr[j] * xr[j];
    double inv = 1.0 / sqrt(ss / d + eps);
    for (int j = 0; j < d; ++j) out[(size_t)t * d + j] = xr[j] * inv;
  }
  free(xr);
  return 0;
}

/*
 * Pre-norm residual stack with a bf16 residual stream:
 *   n_l     = bf16(RMSNorm(x_l))
 *   x_{l+1} = bf16(x_l + MoE_l(n_l))
 * The MoE output is added in full precision and rounded once with the sum.
 */
int orc_stack_forward(const orc_layer *layers, int n_layers,
                      const uint16_t *x_in, int k, double eps,
                      uint16_t *x_out, int nthreads) {
  if (n_layers < 1 || k < 1) return -1;
  const int d = layers[0].d;
  double *nrm = malloc(sizeof(double) * (size_t)k * d);
  double *moe = malloc(sizeof(double) * (size_t)k * d);
  uint16_t *nb = malloc(sizeof(uint16_t) * (size_t)k * d);
  if (!nrm || !moe || !nb) return -2;
  memcpy(x_out, x_in, sizeof(uint16_t) * (size_t)k * d);
  for (int l = 0; l < n_layers; ++l) {
    if (layers[l].d != d) return -1;
    orc_rmsnorm(x_out, ORC_BF16, k, d, eps, nrm);
    for (size_t i = 0; i < (size_t)k * d; ++i) nb[i] = orc_double_to_bf16(nrm[i]);
    int rc = orc_moe_forward(&layers[l], nb, ORC_BF16, k, moe, nthreads);
    if (rc) return rc;
    for (size_t i = 0; i < (size_t)k * d; ++i)
      x_out[i] = orc_double_to_bf16(orc_bf16_to_double(x_out[i]) + moe[i]);
  }
  free(nrm);
  free(moe);
  free(nb);
  return 0;
}

/* ------------------------------------------------------------------ */
/* greedy acceptance                                                   */
/* ------------------------------------------------------------------ */

/* a[i] = argmax_v logits[i][v]; equal values go to the lowest v. */
int orc_argmax_rows(const void *logits, int dtype, int rows, int V,
                    int32_t *a) {
  if (!act_ok(dtype) || rows < 1 || V < 1) return -1;
  double *row = malloc(sizeof(double) * V);
  if (!row) return -2;
  for (int i = 0; i < rows; ++i) {
    orc_decode_rows(dtype, logits, NULL, i, 1, V, row);
    int best = 0;
    for (int v = 1; v < V; ++v)
      if (row[v] > row[best]) best = v;
    a[i] = best;
  }
  free(row);
  return 0;
}

/*
 * Greedy verification ([P1] "Speculative decoding": the target only accepts
 * tokens it would have produced itself, and a cycle commits the accepted
 * draft prefix plus one token of the target's own; [P2] "Why drafter
 * performance doesn't really matter": the nth drafted token is accepted only
 * if the n-1 before it were).
 *   a = row-wise argmax of logits[k+1][V]
 *   n = number of leading positions i < k with draft[i] == a[i]
 *   tau = n + 1;  committed[0..tau-1] = a[0..tau-1], committed[tau..k] = -1
 */
int orc_accept_greedy(const void *logits, int dtype, int k, int V,
                      const int32_t *draft, int32_t *tau,
                      int32_t *committed) {
  if (k < 0 || V < 1) return -1;
  int32_t *a = malloc(sizeof(int32_t) * (k + 1));
  if (!a) return -2;
  int rc = orc_argmax_rows(logits, dtype, k + 1, V, a);
  if (rc) return rc;
  int n = 0;
  while (n < k && draft[n] == a[n]) ++n;
  *tau = n + 1;
  if (committed)
    for (int i = 0; i <= k; ++i) committed[i] = (i <= n) ? a[i] : -1;
  free(a);
  return 0;
}

int orc_num_threads_available(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}
