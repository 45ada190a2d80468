/* A C caller on the GPU: device buffers from the CUDA runtime, a paged
 * bf16 cache with a shuffled block table, decode_attn() and
 * decode_attn_host() on the same inputs.  Their outputs must be identical bit
 * for bit and finite, with no status bit set.  Prints "ok" and exits 0, or
 * names the first failed check and exits 1. */
#include <stdio.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <cuda_runtime.h>

#include "decode_attn.h"

#define CHECK(cond)                                            \
  do {                                                         \
    if (!(cond)) {                                             \
      printf("failed: %s (line %d)\n", #cond, __LINE__);      \
      return 1;                                                \
    }                                                          \
  } while (0)

static uint32_t lcg_state = 12345u;
static uint32_t lcg(void) {
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return lcg_state;
}
/* bf16 bits of a value in about [-1, 1] */
static uint16_t rand_bf16(void) {
  float f = ((float)(lcg() >> 8) / 16777216.0f) * 2.0f - 1.0f;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int main(void) {
  const int B = 3, T = 4, Hq = 16, Hkv = 4, D = DECODE_ATTN_HEAD_DIM, page = 16;
  const int lens[3] = {700, 35, 1201};
  const int max_len = 1216, max_pages = max_len / page;
  int num_pages = 0;
  for (int b = 0; b < B; ++b) num_pages += (lens[b] + page - 1) / page;
  const size_t q_elems = (size_t)B * T * Hq * D;
  const size_t kv_elems = (size_t)num_pages * page * Hkv * D;
  const size_t rows = (size_t)B * T * Hq;

  /* host inputs: random q / K / V, pages handed out in a shuffled order */
  uint16_t* q = malloc(q_elems * 2);
  uint16_t* kv = malloc(kv_elems * 2 * 2);
  int32_t* bt = malloc((size_t)B * max_pages * 4);
  int32_t* perm = malloc((size_t)num_pages * 4);
  CHECK(q && kv && bt && perm);
  for (size_t i = 0; i < q_elems; ++i) q[i] = rand_bf16();
  for (size_t i = 0; i < 2 * kv_elems; ++i) kv[i] = rand_bf16();
  for (int i = 0; i < num_pages; ++i) perm[i] = i;
  for (int i = num_pages - 1; i > 0; --i) {
    const int j = (int)(lcg() % (uint32_t)(i + 1));
    const int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  for (int b = 0, used = 0; b < B; ++b)
    for (int p = 0; p < max_pages; ++p)
      bt[b * max_pages + p] = p < (lens[b] + page - 1) / page ? perm[used++] : -1;

  decode_attn_params prm;
  decode_attn_params_init(&prm, B, T, Hq, Hkv, D, page, max_pages, num_pages, max_len, 1);
  int32_t splits = 0, chunk = 0;
  CHECK(decode_attn_plan(&prm, lens, &splits, &chunk) == DA_OK && splits >= 1);
  size_t ws_bytes = 0, host_ws_bytes = 0;
  CHECK(decode_attn_workspace_bytes(&prm, splits, &ws_bytes) == DA_OK);
  CHECK(decode_attn_host_workspace_bytes(&prm, splits, &host_ws_bytes) == DA_OK);

  void *d_q, *d_k, *d_v, *d_out, *d_ws, *d_hws;
  int32_t *d_bt, *d_lens, *d_status;
  float* d_lse;
  CHECK(cudaMalloc(&d_q, q_elems * 2) == cudaSuccess);
  CHECK(cudaMalloc(&d_k, kv_elems * 2) == cudaSuccess);
  CHECK(cudaMalloc(&d_v, kv_elems * 2) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_bt, (size_t)B * max_pages * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_lens, B * 4) == cudaSuccess);
  CHECK(cudaMalloc(&d_out, q_elems * 2) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_lse, rows * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_status, 4) == cudaSuccess);
  CHECK(cudaMalloc(&d_ws, ws_bytes > 0 ? ws_bytes : 16) == cudaSuccess);
  CHECK(cudaMalloc(&d_hws, host_ws_bytes) == cudaSuccess);
  CHECK(cudaMemcpy(d_q, q, q_elems * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(d_k, kv, kv_elems * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(d_v, kv + kv_elems, kv_elems * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(d_bt, bt, (size_t)B * max_pages * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(d_lens, lens, B * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemset(d_status, 0, 4) == cudaSuccess);

  /* device entry */
  CHECK(decode_attn(&prm, d_q, d_k, d_v, d_bt, d_lens, d_out, d_lse, splits, d_ws, ws_bytes,
                    d_status, NULL) == DA_OK);
  uint16_t* out1 = malloc(q_elems * 2);
  float* lse1 = malloc(rows * 4);
  int32_t status1 = -1;
  CHECK(out1 && lse1);
  CHECK(cudaMemcpy(out1, d_out, q_elems * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(lse1, d_lse, rows * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(&status1, d_status, 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(status1 == 0);

  /* host-buffer entry, same inputs and split count */
  uint16_t* out2 = malloc(q_elems * 2);
  float* lse2 = malloc(rows * 4);
  int32_t status2 = -1;
  CHECK(out2 && lse2);
  CHECK(decode_attn_host(&prm, q, d_k, d_v, bt, lens, out2, lse2, splits, d_hws, host_ws_bytes,
                         &status2, NULL) == DA_OK);
  CHECK(status2 == 0);
  CHECK(memcmp(out1, out2, q_elems * 2) == 0);
  CHECK(memcmp(lse1, lse2, rows * 4) == 0);
  for (size_t i = 0; i < q_elems; ++i) CHECK(isfinite(bf16_to_float(out1[i])));
  for (size_t i = 0; i < rows; ++i) CHECK(isfinite(lse1[i]));

  cudaFree(d_q); cudaFree(d_k); cudaFree(d_v); cudaFree(d_bt); cudaFree(d_lens);
  cudaFree(d_out); cudaFree(d_lse); cudaFree(d_status); cudaFree(d_ws); cudaFree(d_hws);
  free(q); free(kv); free(bt); free(perm); free(out1); free(lse1); free(out2); free(lse2);
  printf("ok\n");
  return 0;
}
