/* A plain C caller of librpa (include/rpa.h), host paths only: workspace
 * sizing, refusal codes, status strings and misaligned-pointer refusal.
 * Compiled and run by tests/test_c_caller.py; exits 0 when every check holds
 * and prints the first one that does not. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "rpa.h"

static rpa_params_t decode_params(void) {
  rpa_params_t p;
  memset(&p, 0, sizeof p);
  p.num_q_heads = 32;
  p.num_kv_heads = 8;
  p.head_dim = 128;
  p.page_size = 16;
  p.num_pages = 80000;
  p.pages_per_seq = 256;
  p.max_num_seqs = 256;
  p.total_tokens = 256;
  p.kv_dtype = RPA_KV_BF16;
  p.softmax_scale = 0.08838835f;
  p.k_scale = 1.0f;
  p.v_scale = 1.0f;
  return p;
}

#define CHECK(cond, what)                   \
  do {                                      \
    if (!(cond)) {                          \
      printf("failed: %s\n", what);        \
      return 1;                             \
    }                                       \
  } while (0)

int main(void) {
  rpa_params_t p = decode_params();
  size_t bytes = 0;
  CHECK(rpa_workspace_size(&p, &bytes) == RPA_OK && bytes > 0, "workspace size");

  p.head_dim = 80;
  CHECK(rpa_workspace_size(&p, &bytes) == RPA_ERR_UNSUPPORTED, "head_dim 80 refused");
  p = decode_params();
  p.softmax_scale = 0.0f;
  CHECK(rpa_workspace_size(&p, &bytes) == RPA_ERR_INVALID_ARG, "zero softmax scale refused");
  p = decode_params();
  p.kv_dtype = RPA_KV_FP8_E4M3;
  p.head_dim = 96;
  p.page_size = 1;
  CHECK(rpa_workspace_size(&p, &bytes) == RPA_ERR_UNSUPPORTED, "fp8 head_dim 96 on 1-row pages");
  CHECK(rpa_workspace_size(NULL, &bytes) == RPA_ERR_INVALID_ARG, "null params refused");

  /* valid params, one misaligned pointer: refused before any CUDA call */
  p = decode_params();
  char* base = (char*)(uintptr_t)(1u << 20);
  void* ws = (void*)(uintptr_t)(1u << 21);
  const int32_t* i32 = (const int32_t*)base;
  CHECK(rpa_forward(&p, base + 8, base, base, base, i32, i32, i32, i32, NULL, base, ws,
                    (size_t)1 << 40, NULL) == RPA_ERR_INVALID_ARG,
        "misaligned queries refused");
  CHECK(rpa_update_cache(&p, base, base, base, (const int32_t*)(base + 2), i32, i32, i32, ws,
                         (size_t)1 << 40, NULL) == RPA_ERR_INVALID_ARG,
        "misaligned kv_lens refused");

  for (int code = 0; code <= 4; ++code) {
    const char* s = rpa_status_string(code);
    CHECK(s != NULL && s[0] != '\0', "status string");
  }
  printf("ok\n");
  return 0;
}
