/* The fp64 oracle (oracle/cpattn_oracle.c) under AddressSanitizer and
 * UndefinedBehaviorSanitizer, built and run by tests/test_sanitize_cpu.py.
 * Small causal and unmasked cases with ragged shapes, GQA, empty rows and
 * bad arguments; results are checked against properties that hold exactly
 * (constant V, chunked-then-merged equals unchunked) so that the run also
 * exercises every branch.  Exits non-zero on a failed check. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int cpattn_oracle_attention(const float *q, const int64_t *q_pos, int64_t nq, const float *k,
                            const float *v, int64_t kv_pos0, int64_t Skv, int64_t B, int64_t Hq,
                            int64_t Hkv, int64_t D, int causal, double scale, double *o,
                            double *lse, int n_threads);
int cpattn_oracle_merge(const double *o_parts, const double *lse_parts, int64_t n_parts,
                        int64_t rows, int64_t D, double *o, double *lse);

static int failures = 0;
#define EXPECT(cond, what)                           \
  do {                                               \
    if (!(cond)) {                                   \
      printf("FAIL %s (line %d)\n", what, __LINE__); \
      ++failures;                                    \
    }                                                \
  } while (0)

static uint64_t rng_state = 88172645463325252ull;
static float frand(void) { /* xorshift64, uniform in [-1, 1) */
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 7;
  rng_state ^= rng_state << 17;
  return (float)((double)(rng_state >> 11) / 9007199254740992.0 * 2.0 - 1.0);
}

int main(void) {
  const int64_t B = 2, nq = 37, Skv = 53, Hq = 6, Hkv = 2, D = 16, base = 20;
  float *q = malloc(sizeof(float) * B * nq * Hq * D);
  float *k = malloc(sizeof(float) * B * Skv * Hkv * D);
  float *v = malloc(sizeof(float) * B * Skv * Hkv * D);
  int64_t *pos = malloc(sizeof(int64_t) * nq);
  double *o = malloc(sizeof(double) * B * nq * Hq * D), *lse = malloc(sizeof(double) * B * Hq * nq);
  double *o1 = malloc(sizeof(double) * B * nq * Hq * D), *l1 = malloc(sizeof(double) * B * Hq * nq);
  double *parts = malloc(sizeof(double) * 2 * nq * D), *lparts = malloc(sizeof(double) * 2 * nq);
  double *om = malloc(sizeof(double) * nq * D), *lm = malloc(sizeof(double) * nq);
  for (int64_t i = 0; i < B * nq * Hq * D; ++i) q[i] = frand();
  for (int64_t i = 0; i < B * Skv * Hkv * D; ++i) {
    k[i] = frand();
    v[i] = frand();
  }
  for (int64_t i = 0; i < nq; ++i) pos[i] = base - 25 + i; /* the first rows see no key */
  for (int causal = 0; causal <= 1; ++causal) {
    EXPECT(cpattn_oracle_attention(q, pos, nq, k, v, 0, Skv, B, Hq, Hkv, D, causal, 0.25, o, lse, 1) == 0,
           "attention status");
    for (int64_t i = 0; i < B * nq * Hq * D; ++i) EXPECT(isfinite(o[i]), "finite O");
    /* chunked: keys [0, 30) and [30, Skv), merged, equal the whole */
    const int64_t cut = 30;
    double *oa = malloc(sizeof(double) * B * nq * Hq * D), *la = malloc(sizeof(double) * B * Hq * nq);
    double *ob = malloc(sizeof(double) * B * nq * Hq * D), *lb = malloc(sizeof(double) * B * Hq * nq);
    float *ka = malloc(sizeof(float) * B * cut * Hkv * D), *va = malloc(sizeof(float) * B * cut * Hkv * D);
    float *kb = malloc(sizeof(float) * B * (Skv - cut) * Hkv * D);
    float *vb = malloc(sizeof(float) * B * (Skv - cut) * Hkv * D);
    for (int64_t b = 0; b < B; ++b)
      for (int64_t j = 0; j < Skv; ++j)
        for (int64_t t = 0; t < Hkv * D; ++t) {
          const int64_t src = (b * Skv + j) * Hkv * D + t;
          if (j < cut) {
            ka[(b * cut + j) * Hkv * D + t] = k[src];
            va[(b * cut + j) * Hkv * D + t] = v[src];
          } else {
            kb[(b * (Skv - cut) + j - cut) * Hkv * D + t] = k[src];
            vb[(b * (Skv - cut) + j - cut) * Hkv * D + t] = v[src];
          }
        }
    EXPECT(cpattn_oracle_attention(q, pos, nq, ka, va, 0, cut, B, Hq, Hkv, D, causal, 0.25, oa, la, 1) == 0,
           "part a");
    EXPECT(cpattn_oracle_attention(q, pos, nq, kb, vb, cut, Skv - cut, B, Hq, Hkv, D, causal, 0.25, ob, lb,
                                   1) == 0,
           "part b");
    for (int64_t b = 0; b < B; ++b)
      for (int64_t h = 0; h < Hq; ++h) {
        for (int64_t i = 0; i < nq; ++i) {
          lparts[i] = la[(b * Hq + h) * nq + i];
          lparts[nq + i] = lb[(b * Hq + h) * nq + i];
          for (int64_t t = 0; t < D; ++t) {
            parts[i * D + t] = oa[((b * nq + i) * Hq + h) * D + t];
            parts[(nq + i) * D + t] = ob[((b * nq + i) * Hq + h) * D + t];
          }
        }
        EXPECT(cpattn_oracle_merge(parts, lparts, 2, nq, D, om, lm) == 0, "merge status");
        for (int64_t i = 0; i < nq; ++i) {
          const double ref = lse[(b * Hq + h) * nq + i];
          EXPECT((isinf(ref) && isinf(lm[i])) || fabs(lm[i] - ref) < 1e-12, "merged LSE");
          for (int64_t t = 0; t < D; ++t)
            EXPECT(fabs(om[i * D + t] - o[((b * nq + i) * Hq + h) * D + t]) < 1e-12, "merged O");
        }
      }
    free(oa); free(la); free(ob); free(lb); free(ka); free(va); free(kb); free(vb);
  }
  /* constant V: O equals the constant on every row with a visible key */
  for (int64_t i = 0; i < B * Skv * Hkv * D; ++i) v[i] = 0.75f;
  EXPECT(cpattn_oracle_attention(q, pos, nq, k, v, 0, Skv, B, Hq, Hkv, D, 1, 0.25, o1, l1, 2) == 0,
         "constant V status");
  for (int64_t b = 0; b < B; ++b)
    for (int64_t i = 0; i < nq; ++i)
      for (int64_t h = 0; h < Hq; ++h) {
        const int visible = pos[i] >= 0;
        for (int64_t t = 0; t < D; ++t) {
          const double x = o1[((b * nq + i) * Hq + h) * D + t];
          EXPECT(visible ? fabs(x - 0.75) < 1e-12 : x == 0.0, "constant V");
        }
        EXPECT(visible ? isfinite(l1[(b * Hq + h) * nq + i]) : isinf(l1[(b * Hq + h) * nq + i]),
               "empty-row LSE");
      }
  /* bad arguments */
  EXPECT(cpattn_oracle_attention(NULL, pos, nq, k, v, 0, Skv, B, Hq, Hkv, D, 1, 0.25, o, lse, 1) != 0,
         "null q");
  EXPECT(cpattn_oracle_attention(q, pos, nq, k, v, 0, Skv, B, 5, Hkv, D, 1, 0.25, o, lse, 1) != 0,
         "hq not a multiple of hkv");
  EXPECT(cpattn_oracle_merge(NULL, lparts, 2, nq, D, om, lm) != 0, "merge null");
  free(q); free(k); free(v); free(pos); free(o); free(lse); free(o1); free(l1);
  free(parts); free(lparts); free(om); free(lm);
  printf("%s (%d failures)\n", failures ? "FAIL" : "ok", failures);
  return failures ? 1 : 0;
}
