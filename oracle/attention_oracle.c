/*
 * attention_oracle.c -- plain fp64 CPU attention, TEST INFRASTRUCTURE ONLY.
 *
 * This file is the correctness oracle for the GPU FlashAttention-2 forward.
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does.  It shares no code, header or
 * constant with the CUDA sources.
 *
 * What it computes is the plain definition of scaled dot-product attention
 * that the FlashAttention-2 forward reaches exactly (up to rounding order):
 *
 *   s_ij   = scale * sum_k Q[i,k] K[j,k]        for every visible key j
 *   LSE_i  = log sum_j exp(s_ij)                (natural log)
 *   O[i,:] = sum_j exp(s_ij - LSE_i) V[j,:]
 *
 * Sources:
 *  - "Extend Thunder with CUDA-Python", section "Extend Thunder with
 *    CUDA-Python", function flash_attention_reference: the forward is
 *    softmax(scale * Q K^T) V over the SDPA layout [batch..., N, d]; the second
 *    output is L = m + log(l), the natural-log log-sum-exp of the scaled
 *    scores; the default scale is 1/sqrt(d); with is_causal the key index j
 *    is visible to query row i only when i >= j (query and key rows both
 *    counted from 0, i.e. top-left alignment when N_q != N_k).
 *  - "Blackwell Attention Example", section "Attention Kernel Implementation",
 *    docstring of blackwell_attention_kernel: Attention(Q,K,V) =
 *    softmax(Q K^T * scale) V with Q [..., seq_q, d] and K, V [..., seq_k, d];
 *    the same section's blackwell_attention takes V with a head dim Dv of its
 *    own (Q and K share d) and returns O with Dv columns.
 *
 * The evaluation is untiled: for each requested query row all visible scores
 * are formed in fp64, their maximum m is taken, and l = sum exp(s - m);
 * then O = sum exp(s - m) V / l and LSE = m + log(l).  Subtracting m is the
 * usual exact rewriting of the softmax (it cancels in the ratio) and keeps
 * exp() in range; it is not the tiled online-softmax of the method.
 *
 * Inputs are fp32 arrays (every bf16 and fp32 value the GPU sees is exactly
 * representable in fp32); all arithmetic is fp64.  Rows are independent and
 * are spread over OpenMP threads when the library is built with -fopenmp.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * Visible keys of query row i: all N_k keys; with is_causal = 1 (top-left
 * alignment) keys j <= i; with is_causal = 2 (bottom-right alignment, the
 * last query row sees the last key) keys j <= i + N_k - N_q.  The result is a
 * prefix 0 .. n_vis-1 of the keys, possibly empty (bottom-right with
 * N_q > N_k): a row that sees no key has O = 0 and LSE = -inf (an empty sum).
 */
static int64_t visible_keys(int64_t i, int64_t N_q, int64_t N_k, int is_causal) {
  int64_t n = N_k;
  if (is_causal == 1) n = i + 1;
  if (is_causal == 2) n = i + 1 + N_k - N_q;
  if (n > N_k) n = N_k;
  if (n < 0) n = 0;
  return n;
}

/* Number of threads the parallel loop below uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * One (batch, head) slice.
 *   Q: N_q rows of d floats, row i at Q + i*q_row_stride (elements).
 *   K: N_k rows of d floats, row j at K + j*k_row_stride.
 *   V: N_k rows of d_v floats, row j at V + j*v_row_stride.
 *   rows[0..n_rows): the query rows to evaluate (NULL = all N_q rows in order).
 *   O: n_rows x d_v doubles, row r at O + r*d_v.   LSE: n_rows doubles.
 * Returns 0 on success, -1 on bad arguments, -2 if scratch allocation failed.
 */
int oracle_attention_slice_v(const float* Q, int64_t q_row_stride,
                             const float* K, int64_t k_row_stride,
                             const float* V, int64_t v_row_stride,
                             int64_t N_q, int64_t N_k, int64_t d, int64_t d_v,
                             double scale, int is_causal,
                             const int64_t* rows, int64_t n_rows,
                             double* O, double* LSE) {
  if (!Q || !K || !V || !O || !LSE || N_q < 0 || N_k <= 0 || d <= 0 || d_v <= 0 || n_rows < 0 ||
      is_causal < 0 || is_causal > 2)
    return -1;
  if (!rows && n_rows != N_q) return -1;
  int failed = 0;

#pragma omp parallel
  {
    double* s = (double*)malloc((size_t)N_k * sizeof(double));
    if (!s) {
#pragma omp atomic write
      failed = 2;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!s) continue;
      int64_t i = rows ? rows[r] : r;
      double* o = O + r * d_v;
      if (i < 0 || i >= N_q) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      const int64_t n_vis = visible_keys(i, N_q, N_k, is_causal);
      if (n_vis == 0) { /* no visible key: empty sum */
        for (int64_t c = 0; c < d_v; ++c) o[c] = 0.0;
        LSE[r] = -INFINITY;
        continue;
      }

      const float* q = Q + i * q_row_stride;
      double m = -INFINITY;
      for (int64_t j = 0; j < n_vis; ++j) {
        const float* k = K + j * k_row_stride;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int64_t c = 0; c < d_v; ++c) o[c] = 0.0;
      for (int64_t j = 0; j < n_vis; ++j) {
        double p = exp(s[j] - m);
        const float* v = V + j * v_row_stride;
        l += p;
        for (int64_t c = 0; c < d_v; ++c) o[c] += p * (double)v[c];
      }
      for (int64_t c = 0; c < d_v; ++c) o[c] /= l;
      LSE[r] = m + log(l);
    }
    free(s);
  }
  return failed == 1 ? -1 : (failed == 2 ? -2 : 0);
}

/* oracle_attention_slice_v with V of the same head dim as Q and K. */
int oracle_attention_slice(const float* Q, int64_t q_row_stride,
                           const float* K, int64_t k_row_stride,
                           const float* V, int64_t v_row_stride,
                           int64_t N_q, int64_t N_k, int64_t d,
                           double scale, int is_causal,
                           const int64_t* rows, int64_t n_rows,
                           double* O, double* LSE) {
  return oracle_attention_slice_v(Q, q_row_stride, K, k_row_stride, V, v_row_stride, N_q, N_k, d, d, scale,
                                  is_causal, rows, n_rows, O, LSE);
}

/*
 * Backward of one (batch, head) slice, fp64, from the plain definition.
 *
 * With P = softmax(scale * Q K^T) (causal: entries with key j > query i are
 * zero), O = P V and an incoming gradient dO of O, the gradients of the
 * scalar sum(dO * O) are ("Blackwell Attention Example", section "Backward
 * Kernel Implementation": the preprocess row sum and the four products of the
 * backward kernel, written here in natural-log form):
 *
 *   dV_j    = sum_i P_ij dO_i
 *   dP_ij   = dO_i . V_j
 *   delta_i = dO_i . O_i                     (= sum_j P_ij dP_ij)
 *   dS_ij   = P_ij (dP_ij - delta_i)
 *   dQ_i    = scale * sum_j dS_ij K_j
 *   dK_j    = scale * sum_i dS_ij Q_i
 *
 * Q, K and dQ, dK have d columns; V, dO and dV have d_v (V with a head dim of
 * its own, as "Blackwell Attention Example" blackwell_attention allows).
 *
 * Untiled: first every query row's max, sum, O and delta (all rows, since dK
 * and dV need them), then dQ for the requested query rows and dK, dV for the
 * requested key rows, each by a plain loop over the other index.
 *   q_rows[0..n_q_rows), k_rows[0..n_k_rows): rows to evaluate (NULL = all).
 *   dQ: n_q_rows x d, dK: n_k_rows x d, dV: n_k_rows x d_v doubles.
 * Returns 0 on success, -1 on bad arguments, -2 if scratch allocation failed.
 */
int oracle_attention_bwd_slice_v(const float* Q, int64_t q_row_stride,
                                 const float* K, int64_t k_row_stride,
                                 const float* V, int64_t v_row_stride,
                                 const float* dO, int64_t do_row_stride,
                                 int64_t N_q, int64_t N_k, int64_t d, int64_t d_v,
                                 double scale, int is_causal,
                                 const int64_t* q_rows, int64_t n_q_rows,
                                 const int64_t* k_rows, int64_t n_k_rows,
                                 double* dQ, double* dK, double* dV) {
  if (!Q || !K || !V || !dO || N_q <= 0 || N_k <= 0 || d <= 0 || d_v <= 0 || n_q_rows < 0 || n_k_rows < 0 ||
      is_causal < 0 || is_causal > 2)
    return -1;
  if ((!q_rows && n_q_rows != N_q) || (!k_rows && n_k_rows != N_k)) return -1;
  if ((n_q_rows > 0 && !dQ) || (n_k_rows > 0 && (!dK || !dV))) return -1;
  for (int64_t r = 0; q_rows && r < n_q_rows; ++r)
    if (q_rows[r] < 0 || q_rows[r] >= N_q) return -1;
  for (int64_t r = 0; k_rows && r < n_k_rows; ++r)
    if (k_rows[r] < 0 || k_rows[r] >= N_k) return -1;

  double* lse = (double*)malloc((size_t)N_q * sizeof(double));
  double* delta = (double*)malloc((size_t)N_q * sizeof(double));
  if (!lse || !delta) {
    free(lse);
    free(delta);
    return -2;
  }
  int failed = 0;

  /* row statistics: LSE_i = log sum_j exp(s_ij), O_i, delta_i = dO_i . O_i */
#pragma omp parallel
  {
    double* s = (double*)malloc((size_t)N_k * sizeof(double));
    double* o = (double*)malloc((size_t)d_v * sizeof(double));
    if (!s || !o) {
#pragma omp atomic write
      failed = 2;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < N_q; ++i) {
      if (!s || !o) continue;
      const int64_t n_vis = visible_keys(i, N_q, N_k, is_causal);
      if (n_vis == 0) { /* no visible key: O = 0, so delta = 0; P = 0 in every product */
        lse[i] = -INFINITY;
        delta[i] = 0.0;
        continue;
      }
      const float* q = Q + i * q_row_stride;
      double m = -INFINITY;
      for (int64_t j = 0; j < n_vis; ++j) {
        const float* k = K + j * k_row_stride;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int64_t c = 0; c < d_v; ++c) o[c] = 0.0;
      for (int64_t j = 0; j < n_vis; ++j) {
        const double p = exp(s[j] - m);
        const float* v = V + j * v_row_stride;
        l += p;
        for (int64_t c = 0; c < d_v; ++c) o[c] += p * (double)v[c];
      }
      const float* g = dO + i * do_row_stride;
      double dl = 0.0;
      for (int64_t c = 0; c < d_v; ++c) dl += (double)g[c] * (o[c] / l);
      lse[i] = m + log(l);
      delta[i] = dl;
    }
    free(s);
    free(o);
  }

  /* dQ_i = scale * sum_j P_ij (dP_ij - delta_i) K_j */
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < n_q_rows; ++r) {
    if (failed) continue;
    const int64_t i = q_rows ? q_rows[r] : r;
    const int64_t n_vis = visible_keys(i, N_q, N_k, is_causal);
    const float* q = Q + i * q_row_stride;
    const float* g = dO + i * do_row_stride;
    double* out = dQ + r * d;
    for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
      const float* k = K + j * k_row_stride;
      const float* v = V + j * v_row_stride;
      double dot = 0.0, dp = 0.0;
      for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
      for (int64_t c = 0; c < d_v; ++c) dp += (double)g[c] * (double)v[c];
      const double p = exp(scale * dot - lse[i]);
      const double ds = p * (dp - delta[i]);
      for (int64_t c = 0; c < d; ++c) out[c] += scale * ds * (double)k[c];
    }
  }

  /* dV_j = sum_i P_ij dO_i,  dK_j = scale * sum_i dS_ij Q_i  (i sees j) */
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < n_k_rows; ++r) {
    if (failed) continue;
    const int64_t j = k_rows ? k_rows[r] : r;
    const float* k = K + j * k_row_stride;
    const float* v = V + j * v_row_stride;
    double* gk = dK + r * d;
    double* gv = dV + r * d_v;
    for (int64_t c = 0; c < d; ++c) gk[c] = 0.0;
    for (int64_t c = 0; c < d_v; ++c) gv[c] = 0.0;
    for (int64_t i = 0; i < N_q; ++i) {
      if (j >= visible_keys(i, N_q, N_k, is_causal)) continue; /* query i does not see key j */
      const float* q = Q + i * q_row_stride;
      const float* g = dO + i * do_row_stride;
      double dot = 0.0, dp = 0.0;
      for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
      for (int64_t c = 0; c < d_v; ++c) dp += (double)g[c] * (double)v[c];
      const double p = exp(scale * dot - lse[i]);
      const double ds = p * (dp - delta[i]);
      for (int64_t c = 0; c < d_v; ++c) gv[c] += p * (double)g[c];
      for (int64_t c = 0; c < d; ++c) gk[c] += scale * ds * (double)q[c];
    }
  }
  free(lse);
  free(delta);
  return failed ? -2 : 0;
}

/* oracle_attention_bwd_slice_v with V and dO of the same head dim as Q and K. */
int oracle_attention_bwd_slice(const float* Q, int64_t q_row_stride,
                               const float* K, int64_t k_row_stride,
                               const float* V, int64_t v_row_stride,
                               const float* dO, int64_t do_row_stride,
                               int64_t N_q, int64_t N_k, int64_t d,
                               double scale, int is_causal,
                               const int64_t* q_rows, int64_t n_q_rows,
                               const int64_t* k_rows, int64_t n_k_rows,
                               double* dQ, double* dK, double* dV) {
  return oracle_attention_bwd_slice_v(Q, q_row_stride, K, k_row_stride, V, v_row_stride, dO, do_row_stride, N_q,
                                      N_k, d, d, scale, is_causal, q_rows, n_q_rows, k_rows, n_k_rows, dQ, dK, dV);
}
