/* Calls libdion3.so from plain C11 through include/dion3.h, on the host paths only (argument
 * validation and size queries, which touch no GPU).  Exits 0 and prints "ok" when every check
 * holds; otherwise prints the failing check and exits 1. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "dion3.h"

static int failures = 0;

static void check(int cond, const char* what) {
  if (!cond) {
    printf("FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  const float abc[15] = {3.4445f, -4.7750f, 2.0315f, 3.4445f, -4.7750f, 2.0315f, 3.4445f, -4.7750f,
                         2.0315f, 3.4445f, -4.7750f, 2.0315f, 3.4445f, -4.7750f, 2.0315f};
  const int restarts[2] = {2, 4};
  float* fake_f = (float*)(size_t)0x10000;
  int32_t* fake_i = (int32_t*)(size_t)0x20000;

  check(dion3_abi_version() == DION3_ABI_VERSION, "abi version");
  check(dion3_k(4096, 1, 4) == 1024, "k of 4096 at f = 1/4");
  check(dion3_k(768, 1, 8) == 96, "k of 768 at f = 1/8");
  check(dion3_k(5, 0, 1) < 0, "f = 0 rejected");
  check(strncmp(dion3_status_str(DION3_EINVAL), "DION3_", 6) == 0, "status string");

  size_t ws = dion3_step_workspace_bytes(2, 64, 128, 1, 4, 1, DION3_FP16, 2);
  check(ws > 0 && ws % 256 == 0, "step workspace query");
  check(dion3_gram_ns_workspace_bytes(2, 64, 128, DION3_BF16, DION3_FP16, 2) > 0, "gram-ns workspace query");

  /* validation fails before anything is enqueued */
  check(dion3_step(1, 64, 128, NULL, fake_f, fake_f, DION3_BF16, 1, 4, 0.95f, 0.01f, 0.0f, 1, 5, abc,
                   restarts, 2, 1e-7f, DION3_FP16, fake_i, fake_f, ws, NULL, NULL) == DION3_EINVAL,
        "step without W");
  check(dion3_step(1, 64, 128, fake_f, fake_f, fake_f, DION3_BF16, 1, 4, 0.95f, 0.01f, 0.0f, 1, 5, abc,
                   restarts, 2, 1e-7f, DION3_FP16, fake_i, NULL, ws, NULL, NULL) == DION3_EWORKSPACE,
        "step without workspace");
  check(dion3_step_carry(1, 64, 128, fake_f, fake_f, fake_f, DION3_BF16, 1, 4, 0.95f, 0.01f, 0.0f, 1, 5, abc,
                         restarts, 2, 1e-7f, DION3_FP16, fake_i, fake_i, INFINITY, 1, fake_f, ws, NULL, NULL,
                         NULL, 0) == DION3_EINVAL,
        "carried decay with an infinite factor");
  check(dion3_decay_rows(1, 8, 8, fake_f, fake_i, 9, 0.9f, NULL) == DION3_EINVAL, "decay of more rows than n");
  check(dion3_decay_rows(0, 8, 8, NULL, NULL, 2, 0.9f, NULL) == DION3_OK, "empty decay");
  check(dion3_sym_gemm(1, -1, 64, fake_f, 64, 4096, NULL, 64, 4096, NULL, 64, 4096, fake_f, 64, 4096, 1.0f, 0.0f,
                       0.0f, DION3_BF16, DION3_BF16, NULL, NULL) == DION3_EINVAL,
        "sym gemm with negative n");

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
