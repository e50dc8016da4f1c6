/*
 * CPU oracle for the fused row-reduction path -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C with fp64 arithmetic.  Every function is the
 * plain definition of what the method computes, written out loop by loop with no
 * blocking, fusion or reordering, so that a reader can check it against the
 * pages by eye.  It shares no code, header, table or constant with the CUDA
 * library and is never linked into it; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Sources (cited by page title and section):
 *   [Stax4]  "Stax (4): GPU Codegen and Dynamic Shapes" (TensorPlay), section 9
 *            (Chinese original and English translation).
 *   [L8]     "CMU 15-779 Lecture 8: ML Compilers Part 1: Tile-based DSLs",
 *            section 3 (fused softmax) and section 12 (exercises).
 *   [HG12]   "hello-gpu Chapter 12: Fusion", sections 12.1 and 12.3.
 *
 * Functions the pages do not define (LayerNorm with Welford statistics, cross
 * entropy with ignore_index, argmax) follow the textbook / PyTorch reading
 * documented beside each function.
 *
 * ORACLE_PLANT: when compiled with -DORACLE_PLANT=k (k >= 1) one deliberate,
 * plausible mistake is planted, so that the pin tests can show they catch it.
 * The shipped oracle is compiled without it (k = 0).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

int oracle_planted(void) { return ORACLE_PLANT; }

/* bf16 bit pattern -> exact value (bf16 is the upper half of an fp32). */
static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------------------
 * Example 1.1: out[x] = sum_r  s * relu(a[x,r] + b[x,r])
 *
 * [Stax4] section 9.2, Listing 9.1 and the text under it: a and b are loaded
 * as fp32, added in fp32 (tmp2), relu is maximum(0, v) with NaN propagation
 * ("PropagateNan.ALL": a NaN input gives a NaN output, matching eager
 * semantics), the result is multiplied by 2.0 in fp32 (tmp6) and summed along
 * the row (tmp10).  The per-element steps are kept in fp32 exactly as the
 * listing types them; the row sum -- the reduction whose order the forms
 * (persistent, looped, split: section 9.4) are free to change -- is taken in
 * fp64 in index order.  The scale s is a parameter (2 in Example 1.1).
 * ---------------------------------------------------------------------- */
static float relu_propagate_nan(float v) {
#if ORACLE_PLANT == 1
  return fmaxf(0.0f, v); /* planted: fmax drops NaN */
#else
  if (isnan(v)) return v;
  return v > 0.0f ? v : 0.0f;
#endif
}

void oracle_relu_add_sum(const float *a, const float *b, int64_t rows, int64_t cols,
                         int64_t lda, int64_t ldb, float scale, double *out) {
  for (int64_t x = 0; x < rows; ++x) {
    double acc = 0.0;
    for (int64_t r = 0; r < cols; ++r) {
#if ORACLE_PLANT == 2
      double v = (double)a[x * lda + r] + (double)b[x * ldb + r]; /* planted: add in fp64 */
      double t = (isnan(v) ? v : (v > 0.0 ? v : 0.0)) * (double)scale;
      acc += t;
#else
      float v = a[x * lda + r] + b[x * ldb + r];
      float t = relu_propagate_nan(v) * scale;
      acc += (double)t;
#endif
    }
    out[x] = acc;
  }
}

/* Sum of squares (Example 6.2 of [Stax4] section 9.4, Listing 9.4: out = sum x*x
 * along the row) and the row L2 norm ([L8] section 12, exercise 1:
 * sqrt(sum x^2), masked lanes filled with 0). */
void oracle_row_sumsq(const float *x, int64_t rows, int64_t cols, int64_t ld, double *out) {
  for (int64_t i = 0; i < rows; ++i) {
    double acc = 0.0;
    for (int64_t r = 0; r < cols; ++r) {
      float v = x[i * ld + r];
      float sq = v * v; /* the listing squares in fp32 (tmp1 = tmp0 * tmp0) */
      acc += (double)sq;
    }
    out[i] = acc;
  }
}

/* Row L2 norm, [L8] section 12, exercise 1: the square root of the row's sum of
 * squares (the same fp32 squares as above), taken in fp64. */
void oracle_row_l2norm(const float *x, int64_t rows, int64_t cols, int64_t ld, double *out) {
  oracle_row_sumsq(x, rows, cols, ld, out);
  for (int64_t i = 0; i < rows; ++i) {
#if ORACLE_PLANT == 10
    out[i] = out[i] / (double)cols; /* planted: mean square instead of the root */
#else
    out[i] = sqrt(out[i]);
#endif
  }
}

/* ------------------------------------------------------------------------
 * Softmax along the row, [Stax4] section 9.5 (the softmax definition and
 * Listing 9.5) and [L8] section 3:
 *     m = max_k x_k,   y_j = exp(x_j - m) / sum_k exp(x_k - m).
 * NaN anywhere in the row makes the max NaN and so the whole row NaN (the pages
 * do not say how max2 treats NaN; the reading here is that NaN propagates
 * through every max, as it does through relu).  Everything else follows from
 * IEEE arithmetic: a +inf entry gives inf - inf = NaN, an all -inf row gives
 * 0/0 = NaN.
 * ---------------------------------------------------------------------- */
void oracle_softmax(const float *x, int64_t rows, int64_t cols, int64_t ld, double *y) {
  for (int64_t i = 0; i < rows; ++i) {
    const float *row = x + i * ld;
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t k = 0; k < cols; ++k) {
      double v = (double)row[k];
      if (isnan(v)) has_nan = 1;
      else if (v > m) m = v;
    }
    if (has_nan) m = NAN;
#if ORACLE_PLANT == 3
    m = 0.0; /* planted: no max subtraction */
#endif
    double d = 0.0;
    for (int64_t k = 0; k < cols; ++k) d += exp((double)row[k] - m);
    for (int64_t k = 0; k < cols; ++k) y[i * cols + k] = exp((double)row[k] - m) / d;
  }
}

/* ------------------------------------------------------------------------
 * The (m, d) monoid of online softmax, [Stax4] section 9.5:
 *   (m1,d1) (+) (m2,d2) = (M, d1*exp(m1-M) + d2*exp(m2-M)),  M = max(m1,m2);
 *   a single element x is (x, 1); the identity is (-inf, 0).
 * Proposition 9.1: (+) is associative and commutative, so any order and any
 * segmentation gives (max, sum exp(x - max)).
 * Reading where the page is silent: when M = -inf (both operands are the
 * identity) exp(-inf - (-inf)) would be NaN; the merge then returns the
 * identity, as the worked frame of [HG12] section 12.4 does with
 * alpha = exp(-inf - 2) = 0.
 * ---------------------------------------------------------------------- */
void oracle_md_merge(double m1, double d1, double m2, double d2, double *m, double *d) {
  if (isnan(m1) || isnan(m2)) {
    *m = NAN;
    *d = NAN;
    return;
  }
  double M = m1 > m2 ? m1 : m2;
  if (M == -INFINITY) {
    *m = -INFINITY;
    *d = 0.0;
    return;
  }
  double s1 = (m1 == -INFINITY) ? 0.0 : exp(m1 - M);
  double s2 = (m2 == -INFINITY) ? 0.0 : exp(m2 - M);
  *m = M;
  *d = d1 * s1 + d2 * s2;
}

/* Fold x[0..n) left to right with (+), starting from the identity. */
void oracle_md_fold(const double *x, int64_t n, double *m, double *d) {
  double cm = -INFINITY, cd = 0.0;
  for (int64_t k = 0; k < n; ++k) oracle_md_merge(cm, cd, x[k], 1.0, &cm, &cd);
  *m = cm;
  *d = cd;
}

/* ------------------------------------------------------------------------
 * Online softmax-weighted row, [HG12] sections 12.1 and 12.3 (also the
 * (m, l, a) triple of [Stax4] section 9.10): state m = -inf, l = 0, a = 0; for
 * each score s_j:  m' = max(m, s_j), alpha = exp(m - m'), beta = exp(s_j - m'),
 * l' = alpha*l + beta,  a' = alpha*a + beta*V_j;  finally O = a / l.
 * Also returns p_j = exp(s_j - m)/l (the materialised probabilities) and the
 * state after every score (trace_* arrays of n, n, n*D entries; may be NULL).
 * ---------------------------------------------------------------------- */
void oracle_online_attn_row(const double *s, const double *V, int64_t n, int64_t D, double *p,
                            double *O, double *trace_m, double *trace_l, double *trace_a,
                            double *trace_alpha, double *trace_beta) {
  double m = -INFINITY, l = 0.0;
  double a[64];
  if (D > 64) return;
  for (int64_t c = 0; c < D; ++c) a[c] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double mn = s[j] > m ? s[j] : m;
    double alpha = (m == -INFINITY) ? 0.0 : exp(m - mn);
    double beta = exp(s[j] - mn);
    l = alpha * l + beta;
    for (int64_t c = 0; c < D; ++c) {
#if ORACLE_PLANT == 4
      a[c] = a[c] + beta * V[j * D + c]; /* planted: old a not rescaled */
#else
      a[c] = alpha * a[c] + beta * V[j * D + c];
#endif
    }
    m = mn;
    if (trace_m) trace_m[j] = m;
    if (trace_l) trace_l[j] = l;
    if (trace_alpha) trace_alpha[j] = alpha;
    if (trace_beta) trace_beta[j] = beta;
    if (trace_a)
      for (int64_t c = 0; c < D; ++c) trace_a[j * D + c] = a[c];
  }
  for (int64_t c = 0; c < D; ++c) O[c] = a[c] / l;
  for (int64_t j = 0; j < n; ++j) p[j] = exp(s[j] - m) / l;
}

/* ------------------------------------------------------------------------
 * LayerNorm over the row.  Not defined on the pages (LayerNorm is only named
 * as an example operator in [L8] section 1); the standard definition is used:
 *   mean = sum x / n,  var = sum (x - mean)^2 / n   (biased),
 *   rstd = 1 / sqrt(var + eps),  y = (x - mean) * rstd * gamma + beta.
 * x is bf16 (decoded exactly), gamma/beta fp32; the statistics are taken by the
 * exact two-pass formula in fp64 (the Welford / Chan merges a kernel may use
 * reach the same value up to rounding).
 * ---------------------------------------------------------------------- */
void oracle_layernorm(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                      const float *gamma, const float *beta, double eps, double *y,
                      double *mean, double *rstd) {
  for (int64_t i = 0; i < rows; ++i) {
    const uint16_t *row = x + i * ld;
    double s = 0.0;
    for (int64_t k = 0; k < cols; ++k) s += bf16_value(row[k]);
    double mu = s / (double)cols;
    double q = 0.0;
    for (int64_t k = 0; k < cols; ++k) {
      double dlt = bf16_value(row[k]) - mu;
      q += dlt * dlt;
    }
#if ORACLE_PLANT == 5
    double var = q / (double)(cols - 1); /* planted: unbiased variance */
#else
    double var = q / (double)cols;
#endif
#if ORACLE_PLANT == 6
    double rs = 1.0 / sqrt(var) + eps; /* planted: eps outside the sqrt */
#else
    double rs = 1.0 / sqrt(var + eps);
#endif
    mean[i] = mu;
    rstd[i] = rs;
    for (int64_t k = 0; k < cols; ++k)
      y[i * cols + k] = (bf16_value(row[k]) - mu) * rs * (double)gamma[k] + (double)beta[k];
  }
}

/* ------------------------------------------------------------------------
 * Log-softmax + cross entropy per row, with ignore_index.
 * The log-sum-exp is LSE = m + log sum_k exp(x_k - m) ([Stax4] section 9.10,
 * "LSE_i = m_i + log l_i"), with (m, l) the row's max and sum of exponentials
 * ([Stax4] section 9.5).  The pages do not define cross entropy; the reading
 * follows PyTorch's cross_entropy(reduction='mean', ignore_index):
 *   loss_row = LSE - x[t]           for 0 <= t < V,
 *   loss_row = 0                    for t == ignore_index (row not counted),
 *   loss_row = NaN, flagged bad     for any other t,
 *   mean = sum of loss_row over rows with t != ignore_index / their count
 *          (NaN when every row is ignored: 0/0).
 * target_logit = x[t] for valid rows, 0 for ignored rows, NaN for bad rows.
 * argmax = first index of the row maximum; a NaN counts as the maximum and the
 * first NaN wins (the pages do not define argmax; lowest index breaks ties).
 * A NaN in the row makes m, LSE and the loss NaN.
 * ---------------------------------------------------------------------- */
/* Logit k of row i, from bf16 bit patterns (f32 == 0) or fp32 values. */
static double logit_value(const void *logits, int f32, int64_t ld, int64_t i, int64_t k) {
  if (f32) return (double)((const float *)logits)[i * ld + k];
  return bf16_value(((const uint16_t *)logits)[i * ld + k]);
}

static void xent_rows(const void *logits, int f32, int64_t rows, int64_t cols, int64_t ld,
                      const int64_t *target, int64_t ignore_index, double *loss, double *lse_out,
                      double *target_logit, int64_t *argmax, double *mean, int64_t *n_counted,
                      int64_t *n_bad) {
  double sum = 0.0;
  int64_t cnt = 0, bad = 0;
  for (int64_t i = 0; i < rows; ++i) {
    double m = -INFINITY;
    int64_t am = 0;
    int has_nan = 0;
    for (int64_t k = 0; k < cols; ++k) {
      double v = logit_value(logits, f32, ld, i, k);
      if (isnan(v)) {
        if (!has_nan) am = k;
        has_nan = 1;
      } else if (!has_nan && v > m) {
        m = v;
        am = k;
      }
#if ORACLE_PLANT == 7
      if (!has_nan && v == m) am = k; /* planted: last index wins ties */
#endif
    }
    if (has_nan) m = NAN;
    double l = 0.0;
    for (int64_t k = 0; k < cols; ++k) l += exp(logit_value(logits, f32, ld, i, k) - m);
#if ORACLE_PLANT == 8
    double lse = log(l); /* planted: max dropped from the LSE */
#else
    double lse = m + log(l);
#endif
    int64_t t = target[i];
    if (lse_out) lse_out[i] = lse;
    if (argmax) argmax[i] = am;
    if (t == ignore_index) {
      loss[i] = 0.0;
      if (target_logit) target_logit[i] = 0.0;
#if ORACLE_PLANT == 9
      ++cnt; /* planted: ignored rows counted in the mean */
#endif
    } else if (t < 0 || t >= cols) {
      loss[i] = NAN;
      if (target_logit) target_logit[i] = NAN;
      ++bad;
      ++cnt;
      sum += NAN;
    } else {
      double xt = logit_value(logits, f32, ld, i, t);
      loss[i] = lse - xt;
      if (target_logit) target_logit[i] = xt;
      ++cnt;
      sum += loss[i];
    }
  }
  if (mean) *mean = sum / (double)cnt; /* 0/0 = NaN when every row is ignored */
  if (n_counted) *n_counted = cnt;
  if (n_bad) *n_bad = bad;
}

/* bf16 logits (bit patterns) */
void oracle_xent(const uint16_t *logits, int64_t rows, int64_t cols, int64_t ld,
                 const int64_t *target, int64_t ignore_index, double *loss, double *lse_out,
                 double *target_logit, int64_t *argmax, double *mean, int64_t *n_counted,
                 int64_t *n_bad) {
  xent_rows(logits, 0, rows, cols, ld, target, ignore_index, loss, lse_out, target_logit, argmax,
            mean, n_counted, n_bad);
}

/* fp32 logits: the same definition on fp32 values */
void oracle_xent_f32(const float *logits, int64_t rows, int64_t cols, int64_t ld,
                     const int64_t *target, int64_t ignore_index, double *loss, double *lse_out,
                     double *target_logit, int64_t *argmax, double *mean, int64_t *n_counted,
                     int64_t *n_bad) {
  xent_rows(logits, 1, rows, cols, ld, target, ignore_index, loss, lse_out, target_logit, argmax,
            mean, n_counted, n_bad);
}
