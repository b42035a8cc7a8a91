/* A C program driving a chunked prefill through include/cp_api.h with the
 * CUDA runtime alone (no Python, no PyTorch): a 300-token GQA prompt (8 query
 * / 2 KV heads x 64, bf16) in chunks of 128 through cp_prefill_chunk.  It
 * writes q, k, v and the output (raw bf16, in that order) to the file named
 * by its argument; tests/test_capi_c.py builds and runs it and compares the
 * output with the oracle. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "cp_api.h"

enum { N = 300, W = 128, HQ = 8, HKV = 2, D = 64, CAP = 384 };

static uint16_t to_bf16(float x) {  /* round to nearest even */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double uniform(uint64_t* s) {  /* xorshift64*, in [-1, 1) */
  *s ^= *s >> 12; *s ^= *s << 25; *s ^= *s >> 27;
  return (double)((*s * 2685821657736338717ull) >> 11) / 4503599627370496.0 - 1.0;
}

#define CHECK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
  printf("cuda error %s at %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

int main(int argc, char** argv) {
  if (argc != 2) return 1;
  static uint16_t q[N * HQ * D], k[N * HKV * D], v[N * HKV * D], o[N * HQ * D];
  uint64_t seed = 0x9E3779B97F4A7C15ull;
  for (int i = 0; i < N * HQ * D; ++i) q[i] = to_bf16((float)uniform(&seed));
  for (int i = 0; i < N * HKV * D; ++i) k[i] = to_bf16((float)uniform(&seed));
  for (int i = 0; i < N * HKV * D; ++i) v[i] = to_bf16((float)uniform(&seed));
  cp_layer_desc desc = {CP_BF16, 1, HQ, HKV, D, CP_CACHE_CONTIG, CAP, 0, 0, 0, 0.f};
  const size_t ws_bytes = cp_workspace_size(&desc, W, CAP, 1);
  void *dq, *dk, *dv, *dout, *kc, *vc, *ws;
  int32_t *lens, *status;
  CHECK(cudaMalloc(&dq, sizeof q)); CHECK(cudaMalloc(&dk, sizeof k)); CHECK(cudaMalloc(&dv, sizeof v));
  CHECK(cudaMalloc(&dout, sizeof o));
  CHECK(cudaMalloc(&kc, (size_t)HKV * CAP * D * 2)); CHECK(cudaMalloc(&vc, (size_t)HKV * CAP * D * 2));
  CHECK(cudaMalloc(&ws, ws_bytes)); CHECK(cudaMemset(ws, 0, ws_bytes));
  CHECK(cudaMalloc((void**)&lens, 4)); CHECK(cudaMemset(lens, 0, 4));
  CHECK(cudaMalloc((void**)&status, 4)); CHECK(cudaMemset(status, 0, 4));
  CHECK(cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dk, k, sizeof k, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dv, v, sizeof v, cudaMemcpyHostToDevice));
  int32_t sizes[8];
  const int32_t nc = cp_chunk_plan(N, W, sizes, 8);
  int32_t past = 0;
  for (int c = 0; c < nc; ++c) {
    const int32_t r = sizes[c];
    const int rc = cp_prefill_chunk(&desc, (char*)dq + (size_t)past * HQ * D * 2, (char*)dk + (size_t)past * HKV * D * 2,
                                    (char*)dv + (size_t)past * HKV * D * 2, kc, vc, lens, NULL, NULL, r, r, past,
                                    (char*)dout + (size_t)past * HQ * D * 2, ws, ws_bytes, status, NULL);
    if (rc != CP_OK) { printf("cp_prefill_chunk: %s\n", cp_status_string(rc)); return 1; }
    past += r;
  }
  CHECK(cudaDeviceSynchronize());
  int32_t hlens = 0, hstatus = 0;
  CHECK(cudaMemcpy(o, dout, sizeof o, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(&hlens, lens, 4, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(&hstatus, status, 4, cudaMemcpyDeviceToHost));
  FILE* f = fopen(argv[1], "wb");
  if (!f || fwrite(q, sizeof q, 1, f) != 1 || fwrite(k, sizeof k, 1, f) != 1 || fwrite(v, sizeof v, 1, f) != 1 ||
      fwrite(o, sizeof o, 1, f) != 1 || fclose(f) != 0) {
    printf("cannot write %s\n", argv[1]);
    return 1;
  }
  printf("chunks %d seqlens_k %d status %d\n", (int)nc, (int)hlens, (int)hstatus);
  return (hlens == N && hstatus == 0) ? 0 : 2;
}
