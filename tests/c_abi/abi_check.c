/* A C99 caller of the decode-attention C ABI (host side only): the public
 * header compiles as plain C, and the library linked into a C program gives
 * the documented answers for dense strides, workspace sizes, the planner
 * for an explicit device shape and argument errors without touching a GPU.  Prints "ok" and exits 0, or names the
 * first failed check and exits 1. */
#include <stdio.h>
#include <string.h>

#include "decode_attn.h"

#define CHECK(cond)                                            \
  do {                                                         \
    if (!(cond)) {                                             \
      printf("failed: %s (line %d)\n", #cond, __LINE__);      \
      return 1;                                                \
    }                                                          \
  } while (0)

int main(void) {
  decode_attn_params p;
  size_t bytes = 0;
  int32_t chunk = 0;
  /* 3 requests, 2 new tokens, 8 query / 2 KV heads, 16-token pages */
  decode_attn_params_init(&p, 3, 2, 8, 2, DECODE_ATTN_HEAD_DIM, 16, 100, 500, 1000, 1);
  CHECK(p.q_stride_head == 128 && p.q_stride_token == 8 * 128 && p.q_stride_batch == 2 * 8 * 128);
  CHECK(p.kv_stride_head == 128 && p.kv_stride_token == 2 * 128 && p.kv_stride_page == 16 * 2 * 128);
  CHECK(p.block_table_stride == 100 && p.flags == 0 && p.k_scale == 1.0f && p.v_scale == 1.0f);

  CHECK(decode_attn_chunk_len(&p, 7, &chunk) == DA_OK && chunk == 144);
  CHECK(decode_attn_workspace_bytes(&p, 1, &bytes) == DA_OK && bytes == 0);
  CHECK(decode_attn_workspace_bytes(&p, 7, &bytes) == DA_OK &&
        bytes == (size_t)(3 * 2 * 8) * 7 * (128 + 1) * 4);
  CHECK(decode_attn_host_workspace_bytes(&p, 7, &bytes) == DA_OK && bytes > 0);
  CHECK(decode_attn_chunk_len(&p, 0, &chunk) == DA_ERR_SPLITS);

  /* the planner for an explicit device shape: B = 1, 32 heads, 128K tokens
   * on 152 SMs x 4 resident CTAs -> one wave of 16 chunks of 8192 tokens */
  {
    decode_attn_params u;
    int32_t splits = 0;
    decode_attn_params_init(&u, 1, 1, 32, 32, DECODE_ATTN_HEAD_DIM, 0, 0, 0, 131072, 0);
    CHECK(decode_attn_plan_slots(&u, NULL, 152 * 4, &splits, &chunk) == DA_OK && splits == 16 &&
          chunk == 8192);
    CHECK(decode_attn_plan_slots(&u, NULL, 0, &splits, &chunk) == DA_ERR_BAD_SHAPE);
  }

  /* argument errors come back before anything is launched */
  CHECK(decode_attn(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL, 0, NULL, NULL) ==
        DA_ERR_NULL_POINTER);
  {
    decode_attn_params bad = p;
    bad.head_dim = 64;
    CHECK(decode_attn_workspace_bytes(&bad, 1, &bytes) == DA_ERR_HEAD_DIM);
    bad = p;
    bad.num_q_heads = 7; /* not a multiple of the KV heads */
    CHECK(decode_attn_workspace_bytes(&bad, 1, &bytes) == DA_ERR_BAD_SHAPE);
  }
  /* an empty batch is a no-op even without buffers */
  {
    decode_attn_params empty;
    decode_attn_params_init(&empty, 0, 1, 8, 2, DECODE_ATTN_HEAD_DIM, 0, 0, 0, 64, 0);
    CHECK(decode_attn(&empty, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL, 0, NULL, NULL) ==
          DA_OK);
  }
  CHECK(strcmp(decode_attn_status_string(DA_OK), "ok") == 0);
  printf("ok\n");
  return 0;
}
