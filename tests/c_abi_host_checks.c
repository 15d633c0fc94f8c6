/*
 * A plain C program against include/spec_verify.h and libspecverify.so: the
 * boundary needs no C++ and no Python. It exercises what runs on the host
 * without a GPU (status strings, workspace sizing and argument validation,
 * which returns before any CUDA call) and prints "ok" when every check holds.
 * Built and run by tests/test_library_abi.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "spec_verify.h"

static int failures = 0;

#define CHECK(cond)                                             \
  do {                                                          \
    if (!(cond)) {                                              \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++failures;                                               \
    }                                                           \
  } while (0)

int main(void) {
  /* status strings */
  CHECK(strcmp(spec_status_string(SPEC_OK), "ok") == 0);
  CHECK(spec_status_string(SPEC_ERR_INVALID_ARG) != NULL);
  CHECK(spec_status_string(12345) != NULL);

  /* workspace sizing: a valid shape needs some bytes, an invalid one none */
  spec_attn_desc d;
  d.batch = 32;
  d.num_q_heads = 32;
  d.num_kv_heads = 8;
  d.head_dim = 128;
  d.block_size = 64;
  d.max_blocks_per_seq = 32;
  d.num_blocks = 32 * 32;
  CHECK(spec_verify_attention_workspace(&d, 3) > 0);
  spec_attn_desc bad = d; /* an invalid descriptor */
  bad.num_kv_heads = 0;
  CHECK(spec_verify_attention_workspace(&bad, 3) == 0);
  spec_attn_desc odd = d; /* a valid descriptor this build has no kernel for */
  odd.head_dim = 96;

  /* kernel plan: 16 packed rows at D = 128 run on mma.sync tiles (no device query) */
  spec_attn_plan plan;
  memset(&plan, 0, sizeof plan);
  CHECK(spec_verify_attention_plan(&d, 3, &plan) == SPEC_OK);
  CHECK(plan.kernel == SPEC_ATTN_KERNEL_MMA && plan.m_tiles == 1 && plan.stages >= 2 && plan.p_buffers == 0);
  CHECK(spec_verify_attention_plan(&d, 3, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(spec_verify_attention_plan(&odd, 3, &plan) == SPEC_ERR_UNSUPPORTED);

  /* argument validation returns before anything reaches the device */
  void* fake = (void*)(uintptr_t)256; /* never dereferenced on these paths */
  int32_t dummy = 0;
  CHECK(spec_verify_attention(NULL, fake, fake, fake, fake, 3, fake, &d, fake, 1 << 20, NULL, NULL) ==
        SPEC_ERR_INVALID_ARG);
  CHECK(spec_verify_attention(fake, fake, fake, fake, fake, 3, fake, &bad, fake, 1 << 20, NULL, NULL) ==
        SPEC_ERR_INVALID_ARG);
  CHECK(spec_verify_attention(fake, fake, fake, fake, fake, 3, fake, &odd, fake, 1 << 20, NULL, NULL) ==
        SPEC_ERR_UNSUPPORTED);
  CHECK(spec_accept(fake, fake, fake, 1, fake, fake, fake, fake, 2, 0, 100, NULL, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(spec_accept(fake, fake, fake, 1, fake, fake, fake, fake, 2, 32, 100, NULL, NULL) == SPEC_ERR_UNSUPPORTED);
  CHECK(spec_accept(fake, fake, fake, 1, fake, fake, fake, fake, 0, 3, 100, NULL, NULL) == SPEC_OK);
  CHECK(spec_commit_state(NULL, fake, fake, 2, 2, 4, 16, NULL, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(spec_commit_state_aligned(fake, fake, fake, 2, 2, 4, 16, 5, SPEC_ALIGN_LAST, NULL, NULL) ==
        SPEC_ERR_INVALID_ARG);
  CHECK(spec_commit_select(fake, fake, fake, 2, 2, 4, 4, 7, NULL, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(spec_gdn_verify(fake, fake, fake, fake, fake, 0.25f, fake, fake, fake, 2, 0, 2, 16, 16, 4,
                        SPEC_ALIGN_TOKEN, &dummy, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(spec_gdn_verify_pooled(fake, fake, fake, fake, fake, 0.25f, fake, 0, fake, fake, fake, 2, 4, 2, 16, 16, 4,
                               SPEC_ALIGN_TOKEN, NULL, NULL) == SPEC_ERR_INVALID_ARG);
  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
