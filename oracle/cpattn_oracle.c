/*
 * cpattn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU definition of what the context-parallel
 * attention path computes, in fp64.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no code,
 * header or constant with the CUDA library; neither includes the other.
 *
 * What it follows:
 *   "Scaling LLM Inference: Innovations in Tensor Parallelism, Context
 *   Parallelism, and Expert Parallelism" (techreport.ngo rewrite), section
 *   "Context Parallelism for Million-Token Contexts", Pass-KV and Pass-Q
 *   bullets: every CP rank ends with attention over the full context, so the
 *   chunked computation must equal plain causal softmax attention.  The same
 *   article (soumitrasaha.com reading notes), section "The communication
 *   bottleneck across all three axes", CP paragraph: ranks pass K/V around a
 *   ring "to accumulate the full attention result".
 *
 * The pages print no formula.  The definition below is the textbook one:
 *   for query row i at absolute position p_i, head h, kv head h / (Hq / Hkv):
 *     V(i)   = { j : 0 <= j < Skv and (not causal or kv_pos0 + j <= p_i) }
 *     s_ij   = scale * sum_t q[i,h,t] * k[j,h/g,t]
 *     LSE_i  = log sum_{j in V(i)} exp(s_ij)          (natural log)
 *     O_i    = sum_{j in V(i)} exp(s_ij - LSE_i) * v[j,h/g,:]
 *     V(i) empty  =>  LSE_i = -inf, O_i = 0
 *   LSE is evaluated as m + log sum exp(s_ij - m) with m = max s_ij, which is
 *   the same number written so that exp does not overflow.
 *
 * The LSE-weighted merge of partial results over disjoint key sets is
 *     LSE = log sum_p exp(LSE_p),   O = sum_p exp(LSE_p - LSE) * O_p
 * which follows from splitting the sum over V(i) above into the parts.
 *
 * Parity of the absolute error scale on real data is not pinned by the pages
 * (they print no numbers for it); the formulas are pinned by the tests in
 * tests/test_oracle.py (brute force, closed forms, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * Causal (or full) softmax attention of a set of query rows against one block
 * of keys/values, in fp64.
 *
 *   q      [B][nq][Hq][D]  float32 (the exact values the GPU sees, widened)
 *   q_pos  [nq]            absolute position of each query row
 *   k, v   [B][Skv][Hkv][D] float32; key row j sits at absolute position kv_pos0 + j
 *   o      [B][nq][Hq][D]  fp64 output
 *   lse    [B][Hq][nq]     fp64 output (natural log)
 * Returns 0 on success, -1 on bad arguments, -2 if scratch memory is short.
 */
int cpattn_oracle_attention(const float *q, const int64_t *q_pos, int64_t nq,
                            const float *k, const float *v, int64_t kv_pos0,
                            int64_t Skv, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t D, int causal, double scale, double *o,
                            double *lse, int n_threads) {
  if (!q || !q_pos || !k || !v || !o || !lse) return -1;
  if (B < 1 || nq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || D < 1) return -1;
  if (Hq % Hkv != 0) return -1;
  const int64_t g = Hq / Hkv;
  const int64_t n_tasks = B * nq * Hq;
  int failed = 0;
#ifdef _OPENMP
  if (n_threads < 1) n_threads = omp_get_max_threads();
#else
  (void)n_threads;
#endif

#pragma omp parallel num_threads(n_threads) reduction(| : failed)
  {
    double *s = (double *)malloc((size_t)(Skv > 0 ? Skv : 1) * sizeof(double));
    double *acc = (double *)malloc((size_t)D * sizeof(double));
    if (!s || !acc) failed = 1;
#pragma omp for schedule(dynamic, 1)
    for (int64_t task = 0; task < n_tasks; ++task) {
      if (!s || !acc) continue;
      const int64_t h = task % Hq;
      const int64_t i = (task / Hq) % nq;
      const int64_t b = task / (Hq * nq);
      const int64_t hk = h / g;
      const float *qi = q + ((b * nq + i) * Hq + h) * D;
      double *oi = o + ((b * nq + i) * Hq + h) * D;
      double *li = lse + (b * Hq + h) * nq + i;

      /* Number of visible keys: all of them, or those at or before p_i. */
      int64_t n_vis = Skv;
      if (causal) {
        int64_t last = q_pos[i] - kv_pos0; /* last visible key row, may be < 0 */
        n_vis = last + 1;
        if (n_vis < 0) n_vis = 0;
        if (n_vis > Skv) n_vis = Skv;
      }
      if (n_vis == 0) {
        for (int64_t t = 0; t < D; ++t) oi[t] = 0.0;
        *li = -INFINITY;
        continue;
      }

      /* Pass 1: logits s_ij and their maximum. */
      double m = -INFINITY;
      for (int64_t j = 0; j < n_vis; ++j) {
        const float *kj = k + ((b * Skv + j) * Hkv + hk) * D;
        double dot = 0.0;
#pragma omp simd reduction(+ : dot)
        for (int64_t t = 0; t < D; ++t) dot += (double)qi[t] * (double)kj[t];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      /* LSE_i = m + log sum exp(s_ij - m). */
      double sum = 0.0;
      for (int64_t j = 0; j < n_vis; ++j) sum += exp(s[j] - m);
      const double L = m + log(sum);
      /* Pass 2: O_i = sum_j exp(s_ij - LSE_i) v_j. */
      for (int64_t t = 0; t < D; ++t) acc[t] = 0.0;
      for (int64_t j = 0; j < n_vis; ++j) {
        const double w = exp(s[j] - L);
        const float *vj = v + ((b * Skv + j) * Hkv + hk) * D;
        for (int64_t t = 0; t < D; ++t) acc[t] += w * (double)vj[t];
      }
      for (int64_t t = 0; t < D; ++t) oi[t] = acc[t];
      *li = L;
    }
    free(s);
    free(acc);
  }
  return failed ? -2 : 0;
}

/*
 * LSE-weighted merge of n_parts partial results over disjoint key sets, fp64.
 *   o_parts   [n_parts][rows][D],  lse_parts [n_parts][rows]
 *   o         [rows][D],           lse       [rows]
 * A part with LSE = -inf contributes nothing; if every part is -inf the row
 * is empty: LSE = -inf, O = 0.
 */
int cpattn_oracle_merge(const double *o_parts, const double *lse_parts,
                        int64_t n_parts, int64_t rows, int64_t D, double *o,
                        double *lse) {
  if (!o_parts || !lse_parts || !o || !lse) return -1;
  if (n_parts < 0 || rows < 0 || D < 1) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int64_t p = 0; p < n_parts; ++p) {
      const double l = lse_parts[p * rows + r];
      if (l > m) m = l;
    }
    double *orow = o + r * D;
    if (m == -INFINITY) {
      for (int64_t t = 0; t < D; ++t) orow[t] = 0.0;
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int64_t p = 0; p < n_parts; ++p) sum += exp(lse_parts[p * rows + r] - m);
    const double L = m + log(sum);
    for (int64_t t = 0; t < D; ++t) orow[t] = 0.0;
    for (int64_t p = 0; p < n_parts; ++p) {
      const double w = exp(lse_parts[p * rows + r] - L);
      const double *op = o_parts + (p * rows + r) * D;
      for (int64_t t = 0; t < D; ++t) orow[t] += w * op[t];
    }
    lse[r] = L;
  }
  return 0;
}
