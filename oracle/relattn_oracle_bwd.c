/*
 * relattn_oracle_bwd.c -- fp64 CPU oracle for the backward pass of Inkling
 * relative attention.
 *
 * TEST INFRASTRUCTURE ONLY: the plain, slow statement of what the GPU backward
 * computes.  It shares no code with the CUDA library (nor with the forward
 * oracle beside it: the logits are recomputed here from the definition).
 *
 * What is differentiated (page "SGLang and Miles Add Day-0 Support for
 * Inkling", section "Customized Efficient Kernels for Train-Inference
 * Consistency", paragraph "Relative attention": the training backend
 * differentiates through the attention scores and through r, while P stays
 * frozen):
 *
 *   l(i,j)  = s_i * (alpha * q_i.k_j + [0 <= i-j < E] * r_i.P[:, i-j])
 *   p(i,j)  = exp(l(i,j) - lse_i)        over the keys row i can see
 *   out_i   = sum_j p(i,j) v_j
 *
 * Given dout, the chain rule through the softmax gives, per row and head,
 *
 *   D_i      = dout_i . out_i
 *   dl(i,j)  = p(i,j) * (dout_i . v_j - D_i)
 *   dq_i     = s_i * alpha * sum_j dl(i,j) k_j
 *   dk_j    += s_i * alpha * dl(i,j) q_i          (summed over rows and heads)
 *   dv_j    += p(i,j) dout_i                       (summed over rows and heads)
 *   dr_i     = sum_{j: 0 <= i-j < E} s_i * dl(i,j) * P[:, i-j]
 *
 * The masks, positions (bottom-right), GQA map and log-scale s_i are the
 * forward oracle's (see relattn_oracle.c).  Every quantity is fp64; the
 * softmax is the two-pass definition (max, then the sum of exponentials).
 *
 * Layouts (row-major): q, dq [Tq, Hq, D]; k, v, dk, dv [Tk, Hkv, D];
 * r, dr [Tq, Hq, r_dim]; P [r_dim, E]; dout [Tq, Hq, D].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define BWD_F64 0
#define BWD_BF16 1

static double bwd_bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double bwd_load(const void *p, size_t idx, int dtype) {
  if (dtype == BWD_BF16) return bwd_bf16_to_double(((const uint16_t *)p)[idx]);
  return ((const double *)p)[idx];
}

static double bwd_log_scale(int64_t pos, double base) {
  if (!(base > 0.0)) return 1.0;
  double s = log((double)(pos + 1)) / log(base);
  return s > 1.0 ? s : 1.0;
}

/* Returns 0 on success, a negative code on invalid arguments.  Outputs are
 * overwritten (zeroed first). */
int relattn_oracle_backward(int dtype, const void *q, const void *k, const void *v,
                            const void *r, const void *P, const void *dout,
                            const int32_t *cu_q, const int32_t *cu_k, int B, int Hq,
                            int Hkv, int D, int r_dim, int E, int window, double alpha,
                            double log_scale_base, double *dq, double *dk, double *dv,
                            double *dr, int n_threads) {
  if (dtype != BWD_F64 && dtype != BWD_BF16) return -1;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -2;
  if (r_dim < 0 || E < 0) return -3;
  if (log_scale_base > 0.0 && !(log_scale_base > 1.0)) return -4;
  for (int b = 0; b < B; ++b) {
    int64_t lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
    if (lq < 0 || lk < lq) return -5;
  }
  const int64_t Tq = B > 0 ? cu_q[B] : 0, Tk = B > 0 ? cu_k[B] : 0;
  memset(dq, 0, sizeof(double) * (size_t)Tq * Hq * D);
  memset(dk, 0, sizeof(double) * (size_t)Tk * Hkv * D);
  memset(dv, 0, sizeof(double) * (size_t)Tk * Hkv * D);
  if (r_dim > 0) memset(dr, 0, sizeof(double) * (size_t)Tq * Hq * r_dim);
  const int group = Hq / Hkv;
  int status = 0;

  /* one task per (sequence, kv head): it owns the dk / dv rows of that pair
   * and the dq / dr rows of the pair's query heads, so tasks never collide */
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t task = 0; task < (int64_t)B * Hkv; ++task) {
    const int b = (int)(task / Hkv), g = (int)(task % Hkv);
    const int64_t lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
    double *l = (double *)malloc((size_t)(lk > 0 ? lk : 1) * sizeof(double));
    double *o = (double *)malloc((size_t)D * sizeof(double));
    if (!l || !o) {
      status = -7;
      free(l);
      free(o);
      continue;
    }
    for (int h = g * group; h < (g + 1) * group; ++h) {
      for (int64_t tq = 0; tq < lq; ++tq) {
        const int64_t t = cu_q[b] + tq;               /* packed query row */
        const int64_t i = (lk - lq) + tq;             /* its position */
        const double s = bwd_log_scale(i, log_scale_base);
        const int64_t j_lo = (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
        const size_t q_off = ((size_t)t * Hq + h) * D;
        const size_t r_off = ((size_t)t * Hq + h) * (size_t)r_dim;
        /* logits of the visible keys, then the two-pass softmax */
        double m = -INFINITY;
        for (int64_t j = j_lo; j <= i; ++j) {
          const size_t k_off = ((size_t)(cu_k[b] + j) * Hkv + g) * D;
          double qk = 0.0;
          for (int e = 0; e < D; ++e) qk += bwd_load(q, q_off + e, dtype) * bwd_load(k, k_off + e, dtype);
          double bias = 0.0;
          if (i - j < E)
            for (int c = 0; c < r_dim; ++c)
              bias += bwd_load(r, r_off + c, dtype) * bwd_load(P, (size_t)c * E + (i - j), dtype);
          l[j - j_lo] = s * (alpha * qk + bias);
          if (l[j - j_lo] > m) m = l[j - j_lo];
        }
        double Z = 0.0;
        for (int64_t j = j_lo; j <= i; ++j) Z += exp(l[j - j_lo] - m);
        const double lse = m + log(Z);
        /* out_i and D_i = dout_i . out_i */
        for (int e = 0; e < D; ++e) o[e] = 0.0;
        for (int64_t j = j_lo; j <= i; ++j) {
          const double p = exp(l[j - j_lo] - lse);
          const size_t v_off = ((size_t)(cu_k[b] + j) * Hkv + g) * D;
          for (int e = 0; e < D; ++e) o[e] += p * bwd_load(v, v_off + e, dtype);
        }
        double Di = 0.0;
        for (int e = 0; e < D; ++e) Di += bwd_load(dout, q_off + e, dtype) * o[e];
        /* the gradients of this row */
        for (int64_t j = j_lo; j <= i; ++j) {
          const double p = exp(l[j - j_lo] - lse);
          const size_t kv_off = ((size_t)(cu_k[b] + j) * Hkv + g) * D;
          double dP = 0.0;
          for (int e = 0; e < D; ++e) dP += bwd_load(dout, q_off + e, dtype) * bwd_load(v, kv_off + e, dtype);
          const double dl = p * (dP - Di);
          for (int e = 0; e < D; ++e) {
            dq[q_off + e] += s * alpha * dl * bwd_load(k, kv_off + e, dtype);
            dk[kv_off + e] += s * alpha * dl * bwd_load(q, q_off + e, dtype);
            dv[kv_off + e] += p * bwd_load(dout, q_off + e, dtype);
          }
          if (i - j < E)
            for (int c = 0; c < r_dim; ++c)
              dr[r_off + c] += s * dl * bwd_load(P, (size_t)c * E + (i - j), dtype);
        }
      }
    }
    free(l);
    free(o);
  }
  return status;
}
