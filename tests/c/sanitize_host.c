/* Host-only entry points of the C ABI under AddressSanitizer and
 * UndefinedBehaviorSanitizer (built and run by tests/test_sanitize_cpu.py).
 * Sweeps the ring plan, critical path, workspace sizes, launch mode and
 * schedule choice over many shapes, and drives every argument-error path of
 * the compute entry points, none of which may reach a CUDA call.  Exits
 * non-zero on the first unexpected status; the sanitizers abort on any
 * memory or undefined-behaviour error. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "cpattn.h"

static int failures = 0;

#define EXPECT(cond, what)                                \
  do {                                                    \
    if (!(cond)) {                                        \
      printf("FAIL %s (line %d)\n", what, __LINE__);      \
      ++failures;                                         \
    }                                                     \
  } while (0)

static cpattn_tensor view(int64_t b, int64_t s, int64_t h, int64_t d, int dtype) {
  cpattn_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = (void *)0x100000;
  t.dtype = dtype;
  t.b = b;
  t.s = s;
  t.h = h;
  t.d = d;
  t.stride_h = d;
  t.stride_s = h * d;
  t.stride_b = s * h * d;
  return t;
}

static void sweep_plans(void) {
  static cpattn_plan_entry entries[4 * 64 * 64];
  const int chunks[] = {1, 2, 3, 4, 5, 8, 16, 32, 64};
  const int64_t bases[] = {0, -300, 1000};
  for (size_t ci = 0; ci < sizeof(chunks) / sizeof(chunks[0]); ++ci) {
    const int n = chunks[ci];
    const int64_t s = 2LL * n * 48;
    for (int mode = CPATTN_PASS_KV; mode <= CPATTN_PASS_Q; ++mode)
      for (int assign = 0; assign <= 1; ++assign)
        for (int causal = 0; causal <= 1; ++causal)
          for (size_t bi = 0; bi < sizeof(bases) / sizeof(bases[0]); ++bi) {
            cpattn_prefill_options o;
            memset(&o, 0, sizeof(o));
            o.assignment = assign;
            o.launch = CPATTN_LAUNCH_DEFAULT;
            int count = -1;
            const cpattn_status st = cpattn_prefill_plan_ex(s, s, bases[bi], n, mode, causal, &o,
                                                            entries, 4 * 64 * 64, &count);
            const int pieces_ok = assign == 0 || (mode == CPATTN_PASS_KV ? 2 * n <= 64 : 4 * n <= 64);
            EXPECT(st == (pieces_ok ? CPATTN_OK : CPATTN_ERR_UNSUPPORTED), "plan status");
            if (st != CPATTN_OK) continue;
            EXPECT(count >= 0, "plan count");
            int small = -1;  /* capacity below the count writes a prefix only */
            EXPECT(cpattn_prefill_plan_ex(s, s, bases[bi], n, mode, causal, &o, entries, 1, &small) ==
                       CPATTN_OK && small == count, "plan with small capacity");
            double step_max[64], critical = -1.0, total = -1.0;
            EXPECT(cpattn_prefill_critical_path(s, s, bases[bi], n, mode, causal, &o, step_max,
                                                &critical, &total) == CPATTN_OK,
                   "critical path");
            EXPECT(critical >= 0.0 && total >= critical - 1e-9, "critical path values");
            cpattn_tensor q = view(2, s, 4, 128, CPATTN_BF16), k = view(2, s, 2, 128, CPATTN_BF16);
            size_t ws = 0;
            for (int lm = CPATTN_LAUNCH_PER_STEP; lm <= CPATTN_LAUNCH_SINGLE_ONCHIP; ++lm) {
              o.launch = lm;
              EXPECT(cpattn_prefill_workspace_size_ex(&q, &k, bases[bi], n, mode, causal, &o, &ws) ==
                         CPATTN_OK, "workspace size");
              int launch = -1;
              EXPECT(cpattn_prefill_launch_mode(&q, &k, bases[bi], n, mode, causal, &o, &launch) ==
                         CPATTN_OK && launch >= 0 && launch != CPATTN_LAUNCH_AUTO &&
                         launch <= CPATTN_LAUNCH_SINGLE_ONCHIP,
                     "launch mode");
            }
            int pick = 0;
            double kvb = -1.0, qb = -1.0;
            EXPECT(cpattn_prefill_choose_mode_ex(&q, &k, bases[bi], n, causal, &o, &pick, &kvb, &qb) ==
                       CPATTN_OK && kvb >= 0.0 && qb >= 0.0,
                   "schedule choice");
            size_t host = 0;
            EXPECT(cpattn_prefill_host_scratch_size(&q, &k, bases[bi], n, mode, causal, CPATTN_BF16,
                                                    &host) == CPATTN_OK,
                   "host scratch size");
            size_t dec = 0;
            cpattn_tensor qd = view(2, 3, 4, 128, CPATTN_BF16);
            EXPECT(cpattn_decode_workspace_size(&qd, &k, bases[bi] + s, n, causal, &dec) ==
                       CPATTN_OK, "decode workspace size");
          }
  }
}

static void argument_errors(void) {
  cpattn_tensor q = view(1, 256, 4, 128, CPATTN_BF16), k = view(1, 256, 2, 128, CPATTN_BF16);
  cpattn_tensor v = k, o = q;
  float *lse = (float *)0x200000;
  /* null tensors and outputs */
  EXPECT(cpattn_partial(NULL, &k, &v, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG, "null q");
  EXPECT(cpattn_partial(&q, &k, &v, 0, 0, 1, 0.f, &o, NULL, NULL) == CPATTN_ERR_INVALID_ARG, "null lse");
  /* unsupported head dim, bad dtype, misaligned pointer, bad strides */
  cpattn_tensor q96 = view(1, 256, 4, 96, CPATTN_BF16), k96 = view(1, 256, 2, 96, CPATTN_BF16);
  cpattn_tensor o96 = q96;
  EXPECT(cpattn_partial(&q96, &k96, &k96, 0, 0, 1, 0.f, &o96, lse, NULL) == CPATTN_ERR_UNSUPPORTED,
         "head dim 96");
  cpattn_tensor qb = q;
  qb.dtype = 7;
  EXPECT(cpattn_partial(&qb, &k, &v, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG, "dtype");
  cpattn_tensor qm = q;
  qm.data = (void *)0x100008;
  EXPECT(cpattn_partial(&qm, &k, &v, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG, "misaligned");
  cpattn_tensor qs = q;
  qs.stride_s = 100;
  EXPECT(cpattn_partial(&qs, &k, &v, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG, "stride");
  cpattn_tensor k3 = view(1, 256, 3, 128, CPATTN_BF16);
  EXPECT(cpattn_partial(&q, &k3, &k3, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG,
         "hq not a multiple of hkv");
  cpattn_tensor kf = k;
  kf.dtype = CPATTN_FP32;
  EXPECT(cpattn_partial(&q, &kf, &kf, 0, 0, 1, 0.f, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG,
         "mixed dtypes");
  EXPECT(cpattn_partial(&q, &k, &v, (int64_t)1 << 40, 0, 1, 0.f, &o, lse, NULL) ==
             CPATTN_ERR_UNSUPPORTED, "offset range");
  /* merge */
  EXPECT(cpattn_merge(&o, NULL, &o, lse, NULL) == CPATTN_ERR_INVALID_ARG, "merge null lse");
  cpattn_tensor o2 = view(1, 255, 4, 128, CPATTN_BF16);
  EXPECT(cpattn_merge(&o, lse, &o2, lse, NULL) == CPATTN_ERR_INVALID_ARG, "merge shape");
  /* prefill: chunks, mode, workspace */
  char ws_probe;
  EXPECT(cpattn_prefill(&q, &k, &v, 0, 3, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_INVALID_ARG, "chunks do not divide");
  EXPECT(cpattn_prefill(&q, &k, &v, 0, 65, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_INVALID_ARG, "too many chunks");
  EXPECT(cpattn_prefill(&q, &k, &v, 0, 4, 3, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_INVALID_ARG, "bad mode");
  EXPECT(cpattn_prefill(&q, &k, &v, 0, 4, CPATTN_PASS_Q, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_WORKSPACE, "missing workspace");
  EXPECT(cpattn_prefill(&q, &k, &v, 0, 4, CPATTN_PASS_Q, 1, 0.f, &o, lse, &ws_probe, 1, NULL) ==
             CPATTN_ERR_WORKSPACE, "small workspace");
  cpattn_prefill_options bad;
  memset(&bad, 0, sizeof(bad));
  bad.launch = 9;
  EXPECT(cpattn_prefill_ex(&q, &k, &v, 0, 4, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, &bad, NULL) ==
             CPATTN_ERR_INVALID_ARG, "bad launch mode");
  bad.launch = CPATTN_LAUNCH_DEFAULT;
  bad.assignment = 5;
  EXPECT(cpattn_prefill_ex(&q, &k, &v, 0, 4, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, &bad, NULL) ==
             CPATTN_ERR_INVALID_ARG, "bad assignment");
  EXPECT(cpattn_prefill_noalloc(&q, &k, &v, 0, 3, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL) ==
             CPATTN_ERR_INVALID_ARG, "noalloc chunks");
  /* decode */
  EXPECT(cpattn_decode(&q, &k, &v, 0, 0, 1, 0.f, &o, lse, NULL, 0, NULL) == CPATTN_ERR_INVALID_ARG,
         "decode zero chunks");
  /* host-buffer entry point: non-contiguous tensors and missing scratch */
  EXPECT(cpattn_prefill_host(&qs, &k, &v, 0, 4, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_INVALID_ARG, "host strides");
  EXPECT(cpattn_prefill_host(&q, &k, &v, 0, 4, CPATTN_PASS_KV, 1, 0.f, &o, lse, NULL, 0, NULL) ==
             CPATTN_ERR_WORKSPACE, "host scratch");
  /* host-only calls with null outputs */
  size_t ws = 0;
  EXPECT(cpattn_prefill_workspace_size(&q, &k, 0, 4, CPATTN_PASS_KV, 1, NULL) == CPATTN_ERR_INVALID_ARG,
         "workspace null out");
  EXPECT(cpattn_prefill_workspace_size(NULL, &k, 0, 4, CPATTN_PASS_KV, 1, &ws) == CPATTN_ERR_INVALID_ARG,
         "workspace null q");
  int n = 0;
  EXPECT(cpattn_prefill_plan(256, 256, 0, 4, CPATTN_PASS_KV, 1, NULL, 5, &n) == CPATTN_ERR_INVALID_ARG,
         "plan null entries");
  EXPECT(cpattn_prefill_critical_path(256, 256, 0, 4, CPATTN_PASS_KV, 1, NULL, NULL, NULL, NULL) ==
             CPATTN_ERR_INVALID_ARG, "critical path null");
  EXPECT(cpattn_prefill_choose_mode_ex(&q, &k, 0, 4, 1, NULL, NULL, NULL, NULL) == CPATTN_ERR_INVALID_ARG,
         "choose null");
  EXPECT(cpattn_profile_begin(0) == CPATTN_ERR_INVALID_ARG, "profile capacity");
  EXPECT(cpattn_profile_end(NULL, 0, NULL) == CPATTN_ERR_INVALID_ARG, "profile not armed");
  for (int s = 0; s <= 6; ++s) EXPECT(cpattn_status_string((cpattn_status)s) != NULL, "status string");
}

int main(void) {
  sweep_plans();
  argument_errors();
  printf("%s (%d failures)\n", failures ? "FAIL" : "ok", failures);
  return failures ? 1 : 0;
}
