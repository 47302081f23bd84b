/* Plain C11 client of libcpattn.so: includes the public header and calls the
 * host-only entry points (no GPU needed).  Prints one line per check; exits
 * non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "cpattn.h"

#define CHECK(cond, what)                          \
  do {                                             \
    if (!(cond)) {                                 \
      printf("FAIL %s\n", what);                   \
      return 1;                                    \
    }                                              \
    printf("ok %s\n", what);                       \
  } while (0)

static cpattn_tensor view(int64_t s, int64_t h) {
  cpattn_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = (void *)0x10000;
  t.dtype = CPATTN_BF16;
  t.b = 1;
  t.s = s;
  t.h = h;
  t.d = 128;
  t.stride_h = 128;
  t.stride_s = h * 128;
  t.stride_b = s * h * 128;
  return t;
}

int main(void) {
  cpattn_plan_entry entries[64];
  int n = 0;
  /* 4 chunks, causal self-prefill: 4 + 3 + 2 + 1 = 10 non-empty pairs. */
  CHECK(cpattn_prefill_plan(256, 256, 0, 4, CPATTN_PASS_KV, 1, entries, 64, &n) == CPATTN_OK,
        "plan status");
  CHECK(n == 10, "plan pairs");
  CHECK(cpattn_prefill_plan(256, 256, 0, 3, CPATTN_PASS_KV, 1, entries, 64, &n) ==
            CPATTN_ERR_INVALID_ARG,
        "plan rejects chunks that do not divide the sequence");

  double step_max[16], critical = 0.0, total = 0.0;
  cpattn_prefill_options zig;
  memset(&zig, 0, sizeof(zig));
  zig.assignment = CPATTN_ASSIGN_ZIGZAG;
  zig.launch = CPATTN_LAUNCH_DEFAULT;
  CHECK(cpattn_prefill_critical_path(4096, 4096, 0, 4, CPATTN_PASS_KV, 1, &zig, step_max, &critical,
                                     &total) == CPATTN_OK,
        "critical path status");
  CHECK(total > 0.0 && critical * 4 >= total * 0.999 && critical * 4 <= total * 1.001,
        "zigzag balances the ring");

  cpattn_tensor q = view(8192, 32), k = view(8192, 8);
  int launch = -1;
  CHECK(cpattn_prefill_launch_mode(&q, &k, 0, 8, CPATTN_PASS_KV, 1, NULL, &launch) == CPATTN_OK,
        "launch mode status");
  CHECK(launch == CPATTN_LAUNCH_SINGLE_ONCHIP, "short Pass-KV items take one on-chip launch");
  CHECK(cpattn_prefill_launch_mode(&q, &k, 0, 8, CPATTN_PASS_Q, 1, NULL, &launch) == CPATTN_OK,
        "launch mode status");
  CHECK(launch == CPATTN_LAUNCH_SINGLE, "short Pass-Q items take one launch");

  size_t ws = 0;
  CHECK(cpattn_prefill_workspace_size(&q, &k, 0, 8, CPATTN_PASS_Q, 1, &ws) == CPATTN_OK && ws > 0,
        "workspace size");
  int mode = 0;
  double kv_bytes = 0.0, q_bytes = 0.0;
  CHECK(cpattn_prefill_choose_mode(&q, &k, 8, &mode, &kv_bytes, &q_bytes) == CPATTN_OK &&
            (mode == CPATTN_PASS_KV || mode == CPATTN_PASS_Q),
        "schedule choice");
  CHECK(strncmp(cpattn_status_string(CPATTN_ERR_TIMEOUT), "CPATTN", 6) == 0, "status string");
  CHECK(strncmp(cpattn_status_string(CPATTN_ERR_DEVICE_CHECK), "CPATTN", 6) == 0, "status string");
  return 0;
}
