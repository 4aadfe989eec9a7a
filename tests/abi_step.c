/* A decode loop written against include/nk.h alone, in plain C: the C ABI's
 * end-to-end cost without Python or ctypes.
 *
 * One sequence (B = 1, T = 1, 24 q-heads over 4 kv-heads, head_dim 256,
 * 64-key pages): a history of CTX0 - 1 tokens is appended, then every step
 * appends the step's K/V row and attends at the grown context, through
 * nk_decode_step_host from one pinned host buffer (inputs in, output and
 * status out, stream wait). Inputs are deterministic (a 32-bit LCG), so runs
 * repeat. After the timed loop the last step is run once more through
 * nk_decode_step on device copies of the same inputs (rewriting the row with
 * the same codes); its output must equal the host path's bit for bit.
 *
 * Prints one JSON line: steps, microseconds per step (host wall clock around
 * each call), the status words and whether the two paths matched.
 * Exit status 0 when every call returned NK_OK, the status words are 0 and
 * the outputs match.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include "nk.h"

enum { B = 1, T = 1, HQ = 24, HKV = 4, D = 256, P = 64, CTX0 = 32768, STEPS = 200, WARM = 20 };

static uint32_t lcg_state = 12345u;
static uint16_t next_bf16(void) {
  /* uniform in [-2, 2), rounded down to bf16 */
  lcg_state = lcg_state * 1664525u + 1013904223u;
  const float x = ((float)(lcg_state >> 8) / 16777216.0f) * 4.0f - 2.0f;
  uint32_t bits;
  memcpy(&bits, &x, 4);
  return (uint16_t)(bits >> 16);
}

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

#define CK(call)                                                        \
  do {                                                                  \
    cudaError_t e_ = (call);                                            \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 2;                                                         \
    }                                                                   \
  } while (0)
#define NK(call)                                                        \
  do {                                                                  \
    int r_ = (call);                                                    \
    if (r_ != NK_OK) {                                                  \
      fprintf(stderr, "nk error %d (%s) at line %d\n", r_, nk_status_string(r_), __LINE__); \
      return 3;                                                         \
    }                                                                   \
  } while (0)

int main(void) {
  const int max_ctx = CTX0 + STEPS + WARM + 1;
  const int max_pages = (max_ctx + P - 1) / P;
  const int num_pages = max_pages;
  const float sm_scale = 0.0625f; /* 1 / sqrt(256) */

  nk_kv_pool pool;
  const size_t pool_bytes = nk_kv_pool_bytes(num_pages, P, HKV, D);
  CK(cudaMalloc(&pool.base_dev, pool_bytes));
  CK(cudaMemset(pool.base_dev, 0, pool_bytes));
  pool.num_pages = num_pages;
  pool.page_size = P;
  pool.num_kv_heads = HKV;
  pool.head_dim = D;

  /* block table: the pages in a fixed shuffled order */
  int32_t* bt_host = (int32_t*)malloc(sizeof(int32_t) * max_pages);
  for (int i = 0; i < max_pages; ++i) bt_host[i] = (int32_t)(((int64_t)i * 7919) % max_pages);
  int32_t* bt_dev;
  CK(cudaMalloc((void**)&bt_dev, sizeof(int32_t) * max_pages));
  CK(cudaMemcpy(bt_dev, bt_host, sizeof(int32_t) * max_pages, cudaMemcpyHostToDevice));
  int32_t* status_dev;
  CK(cudaMalloc((void**)&status_dev, sizeof(int32_t)));
  CK(cudaMemset(status_dev, 0, sizeof(int32_t)));

  /* history: positions 0 .. CTX0 - 2, appended in chunks of 4,096 rows */
  const int hist = CTX0 - 1, chunk = 4096;
  const size_t row_elems = (size_t)HKV * D;
  uint16_t* kh = (uint16_t*)malloc(sizeof(uint16_t) * row_elems * chunk);
  uint16_t* vh = (uint16_t*)malloc(sizeof(uint16_t) * row_elems * chunk);
  void *kd, *vd;
  int32_t *sp_dev, *cu_dev;
  CK(cudaMalloc(&kd, sizeof(uint16_t) * row_elems * chunk));
  CK(cudaMalloc(&vd, sizeof(uint16_t) * row_elems * chunk));
  CK(cudaMalloc((void**)&sp_dev, sizeof(int32_t)));
  CK(cudaMalloc((void**)&cu_dev, 2 * sizeof(int32_t)));
  for (int pos = 0; pos < hist; pos += chunk) {
    const int n = hist - pos < chunk ? hist - pos : chunk;
    for (size_t i = 0; i < row_elems * (size_t)n; ++i) kh[i] = next_bf16();
    for (size_t i = 0; i < row_elems * (size_t)n; ++i) vh[i] = next_bf16();
    const int32_t cu[2] = {0, n};
    CK(cudaMemcpy(kd, kh, sizeof(uint16_t) * row_elems * n, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(vd, vh, sizeof(uint16_t) * row_elems * n, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(sp_dev, &pos, sizeof(int32_t), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(cu_dev, cu, sizeof(cu), cudaMemcpyHostToDevice));
    NK(nk_kv_append(&pool, bt_dev, max_pages, sp_dev, cu_dev, B, n, kd, vd, status_dev, NULL));
  }
  CK(cudaDeviceSynchronize());

  /* one step's buffers: pinned input and output, device staging and output */
  size_t off[6];
  const size_t in_bytes = nk_step_host_layout(B, B * T, T, HQ, HKV, D, off);
  const size_t out_elems = (size_t)B * T * HQ * D;
  const size_t ws_bytes = nk_decode_workspace_bytes(B, T, HQ, HKV, D, 0);
  if (in_bytes == 0 || ws_bytes == 0) return 4;
  uint8_t* in_host;
  uint16_t *out_host, *out_dev;
  int32_t* status_host;
  void *staging, *ws;
  CK(cudaHostAlloc((void**)&in_host, in_bytes, cudaHostAllocDefault));
  CK(cudaHostAlloc((void**)&out_host, sizeof(uint16_t) * out_elems, cudaHostAllocDefault));
  CK(cudaHostAlloc((void**)&status_host, sizeof(int32_t), cudaHostAllocDefault));
  CK(cudaMalloc(&staging, in_bytes));
  CK(cudaMalloc(&ws, ws_bytes));
  CK(cudaMalloc((void**)&out_dev, sizeof(uint16_t) * out_elems));
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

  double total_us = 0.0;
  int ctx = CTX0 - 1;
  int32_t status_or = 0;
  for (int step = 0; step < WARM + STEPS; ++step) {
    /* this step's K/V row at position ctx, Q, and the sequence metadata */
    uint16_t* k = (uint16_t*)(in_host + off[0]);
    uint16_t* v = (uint16_t*)(in_host + off[1]);
    uint16_t* q = (uint16_t*)(in_host + off[2]);
    for (size_t i = 0; i < row_elems; ++i) k[i] = next_bf16();
    for (size_t i = 0; i < row_elems; ++i) v[i] = next_bf16();
    for (size_t i = 0; i < out_elems; ++i) q[i] = next_bf16();
    ((int32_t*)(in_host + off[3]))[0] = ctx;
    ((int32_t*)(in_host + off[4]))[0] = 0;
    ((int32_t*)(in_host + off[4]))[1] = B * T;
    ((int32_t*)(in_host + off[5]))[0] = ctx + 1;
    const double t0 = now_us();
    NK(nk_decode_step_host(&pool, bt_dev, max_pages, B, B * T, T, HQ, sm_scale, max_ctx, 0, in_host, staging, ws,
                           ws_bytes, out_dev, out_host, status_dev, status_host, st));
    const double t1 = now_us();
    if (step >= WARM) total_us += t1 - t0;
    status_or |= *status_host;
    ++ctx;
  }

  /* the last step again through nk_decode_step on device copies of its inputs */
  uint16_t* out_check = (uint16_t*)malloc(sizeof(uint16_t) * out_elems);
  uint16_t* out2_dev;
  CK(cudaMalloc((void**)&out2_dev, sizeof(uint16_t) * out_elems));
  CK(cudaMemcpy(staging, in_host, in_bytes, cudaMemcpyHostToDevice));
  const uint8_t* sb = (const uint8_t*)staging;
  NK(nk_decode_step(&pool, bt_dev, max_pages, (const int32_t*)(sb + off[3]), (const int32_t*)(sb + off[4]), B * T,
                    sb + off[0], sb + off[1], sb + off[2], (const int32_t*)(sb + off[5]), B, T, HQ, sm_scale, max_ctx,
                    0, ws, ws_bytes, out2_dev, status_dev, st));
  CK(cudaStreamSynchronize(st));
  CK(cudaMemcpy(out_check, out2_dev, sizeof(uint16_t) * out_elems, cudaMemcpyDeviceToHost));
  int32_t status_last = 0;
  CK(cudaMemcpy(&status_last, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost));
  const int match = memcmp(out_check, out_host, sizeof(uint16_t) * out_elems) == 0;
  int finite = 1;
  for (size_t i = 0; i < out_elems; ++i)
    if ((out_host[i] & 0x7f80u) == 0x7f80u) finite = 0;

  printf("{\"steps\": %d, \"us_per_step\": %.2f, \"ctx_first\": %d, \"ctx_last\": %d, \"status\": %d, "
         "\"status_after_check\": %d, \"finite\": %s, \"match\": %s}\n",
         STEPS, total_us / STEPS, CTX0 + WARM, CTX0 + WARM + STEPS - 1, (int)status_or, (int)status_last,
         finite ? "true" : "false", match ? "true" : "false");
  return (status_or == 0 && status_last == 0 && match && finite) ? 0 : 1;
}
