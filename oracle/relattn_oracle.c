/*
 * relattn_oracle.c -- fp64 CPU oracle for Inkling relative attention (forward).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  It shares no code, header, table or
 * helper with the CUDA library; only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load it.  No product code path calls it.
 *
 * What it computes (page "SGLang and Miles Add Day-0 Support for Inkling",
 * section "Attention with Relative Positional Embedding", the rel_logits and
 * attention-logit equations; restated in section "Customized Efficient Kernels
 * for Train-Inference Consistency", paragraph "Relative attention"):
 *
 *   rel_logits(t,h,d) = sum_c r[t,h,c] * P[c,d]                 0 <= d < E
 *   l(i,j,h)          = alpha * q_i.k_j + [0 <= i-j < E] * rel_logits(i,h,i-j)
 *
 * Future keys are masked (causal).  Sliding-window layers keep key j only when
 * i - j < window (same page, paragraph "Attention layout").  Full layers may
 * scale q and the relative logits by a length-dependent factor s (same
 * paragraph); the page gives no formula, and this oracle uses
 *   s(i) = max(1, ln(i+1) / ln(base))   (base <= 0: s = 1),
 * which multiplies the whole logit: l' = s * l.
 *
 * Softmax is evaluated in two passes per row, exactly as defined:
 *   m = max_j l_j,  Z = sum_j exp(l_j - m),  lse = m + ln Z,
 *   out = sum_j exp(l_j - lse) * v_j.
 * No tiling, no streaming, no reordering beyond that definition.
 *
 * Positions: query row t of sequence b sits at position Lk_b - Lq_b + t
 * ("bottom-right" alignment), so a decode row equals the matching last row of
 * a prefill over the same sequence.  GQA: query head h reads kv head
 * h / (Hq / Hkv) (the vLLM page, section on attention: all layers use GQA with
 * head size 128).
 *
 * Layouts (row-major, innermost last):
 *   q [Tq, Hq, D], k and v [Tk, Hkv, D], r [Tq, Hq, r_dim], P [r_dim, E]
 *   out [n_sel, Hq, D], lse [n_sel, Hq]   (n_sel = selected query rows)
 * Inputs are either fp64 or bf16 bit patterns (widened to fp64 exactly).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F64 0
#define ORACLE_BF16 1

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_elem(const void *p, size_t idx, int dtype) {
  if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t *)p)[idx]);
  return ((const double *)p)[idx];
}

/* Length-dependent log-scale (stated reading, see file header). */
static double log_scale_factor(int64_t pos, double base) {
  if (!(base > 0.0)) return 1.0;
  double s = log((double)(pos + 1)) / log(base);
  return s > 1.0 ? s : 1.0;
}

int relattn_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Returns 0 on success, a negative code on invalid arguments. */
int relattn_oracle_forward(int dtype, const void *q, const void *k, const void *v,
                           const void *r, const void *P, const int32_t *cu_q,
                           const int32_t *cu_k, int B, int Hq, int Hkv, int D,
                           int r_dim, int E, int window, double alpha,
                           double log_scale_base, const int64_t *sel_rows,
                           int64_t n_sel, double *out, double *lse, int n_threads) {
  if (dtype != ORACLE_F64 && dtype != ORACLE_BF16) return -1;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -2;
  if (r_dim < 0 || E < 0) return -3;
  if (log_scale_base > 0.0 && !(log_scale_base > 1.0)) return -4;
  for (int b = 0; b < B; ++b) {
    int64_t lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
    if (lq < 0 || lk < lq) return -5;
  }
  const int64_t Tq = B > 0 ? cu_q[B] : 0;
  const int64_t n_rows = sel_rows ? n_sel : Tq;
  for (int64_t s = 0; sel_rows && s < n_sel; ++s)
    if (sel_rows[s] < 0 || sel_rows[s] >= Tq) return -6;
  const int group = Hq / Hkv;
  int status = 0;

#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t task = 0; task < n_rows * Hq; ++task) {
    const int64_t sel = task / Hq;
    const int h = (int)(task % Hq);
    const int64_t t = sel_rows ? sel_rows[sel] : sel; /* packed query row */
    /* sequence holding row t */
    int lo_b = 0, hi_b = B - 1;
    while (lo_b < hi_b) {
      int mid = (lo_b + hi_b + 1) / 2;
      if (cu_q[mid] <= t) lo_b = mid; else hi_b = mid - 1;
    }
    const int b = lo_b;
    const int64_t lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
    const int64_t i = (lk - lq) + (t - cu_q[b]); /* query position */
    const int g = h / group;                      /* kv head */
    const double s = log_scale_factor(i, log_scale_base);
    const int64_t j_lo = (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
    const int64_t n_vis = i - j_lo + 1;

    double *logit = (double *)malloc((size_t)n_vis * sizeof(double));
    if (!logit) { status = -7; continue; }
    const size_t q_off = ((size_t)t * Hq + h) * D;
    const size_t r_off = ((size_t)t * Hq + h) * (size_t)r_dim;
    for (int64_t j = j_lo; j <= i; ++j) {
      const size_t k_off = ((size_t)(cu_k[b] + j) * Hkv + g) * D;
      double qk = 0.0;
      for (int e = 0; e < D; ++e) qk += load_elem(q, q_off + e, dtype) * load_elem(k, k_off + e, dtype);
      const int64_t d = i - j;
      double bias = 0.0;
      if (d < E)
        for (int c = 0; c < r_dim; ++c)
          bias += load_elem(r, r_off + c, dtype) * load_elem(P, (size_t)c * E + d, dtype);
      logit[j - j_lo] = s * (alpha * qk + bias);
    }
    double m = -INFINITY;
    for (int64_t n = 0; n < n_vis; ++n) m = logit[n] > m ? logit[n] : m;
    double Z = 0.0;
    for (int64_t n = 0; n < n_vis; ++n) Z += exp(logit[n] - m);
    const double row_lse = m + log(Z);
    double *o = out + ((size_t)sel * Hq + h) * D;
    for (int e = 0; e < D; ++e) o[e] = 0.0;
    for (int64_t j = j_lo; j <= i; ++j) {
      const double w = exp(logit[j - j_lo] - row_lse);
      const size_t v_off = ((size_t)(cu_k[b] + j) * Hkv + g) * D;
      for (int e = 0; e < D; ++e) o[e] += w * load_elem(v, v_off + e, dtype);
    }
    lse[(size_t)sel * Hq + h] = row_lse;
    free(logit);
  }
  return status;
}
