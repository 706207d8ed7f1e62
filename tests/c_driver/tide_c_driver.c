/*
 * Plain-C user of libtide.so: builds the tiny-block layout (N = 4; q,k,v,o
 * [256,256], w1,w3 [704,256], w2 [256,704], norm [250]), runs the
 * reduce-scatter and the placement on device buffers through the C ABI only
 * (no Python, no PyTorch), and checks every output element bit for bit
 * against the CPU oracle.  Inputs are simple integer-hash bf16 values.
 * Exit status 0 on success.  Test program: part of the test suite.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tide.h"
#include "../../oracle/tide_oracle.h"

#define N 4
#define P 8

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s (%s)\n", what, tide_last_error());
  return 1;
}

static uint16_t value(uint32_t k, uint32_t p, uint32_t i) {
  uint32_t h = (k * 2654435761u) ^ (p * 2246822519u) ^ (i * 3266489917u);
  h ^= h >> 15;
  h *= 2246822519u;
  h ^= h >> 13;
  /* bf16 with a random sign and mantissa, exponent in [2^-4, 2^3) */
  return (uint16_t)(((h >> 16) & 0x8000u) | ((0x7Bu + (h & 7u)) << 7) | ((h >> 3) & 0x7Fu));
}

int main(void) {
  const int32_t ndims[P] = {2, 2, 2, 2, 2, 2, 2, 1};
  const int64_t dims[] = {256, 256, 256, 256, 256, 256, 256, 256, 704, 256, 704, 256, 256, 704, 250};
  int64_t d0[P], inner[P], numel[P];
  int pos = 0;
  for (int p = 0; p < P; ++p) {
    d0[p] = dims[pos];
    inner[p] = ndims[p] == 2 ? dims[pos + 1] : 1;
    numel[p] = d0[p] * inner[p];
    pos += ndims[p];
  }
  tide_layout_t lay = NULL;
  if (tide_layout_create(P, ndims, dims, N, &lay) != TIDE_OK) return fail("tide_layout_create");
  int64_t S = 0, offs[P], shard_n[P];
  tide_layout_rank_block_numel(lay, &S);
  for (int p = 0; p < P; ++p) {
    tide_layout_param_offset(lay, p, &offs[p]);
    tide_layout_shard_numel(lay, p, &shard_n[p]);
  }
  int64_t o_offs[P], o_S = 0;
  if (oracle_layout(P, d0, inner, N, 8, o_offs, &o_S) || o_S != S) return fail("layout differs from the oracle");
  for (int p = 0; p < P; ++p)
    if (o_offs[p] != offs[p]) return fail("offset differs from the oracle");

  /* host inputs and device buffers */
  uint16_t* hg[N * P];
  const uint16_t* dg[N * P];
  float* ds[N * P];
  uint16_t* dp[P];
  for (int k = 0; k < N; ++k)
    for (int p = 0; p < P; ++p) {
      uint16_t* h = malloc(sizeof(uint16_t) * numel[p]);
      for (int64_t i = 0; i < numel[p]; ++i) h[i] = value(k, p, (uint32_t)i);
      hg[k * P + p] = h;
      void* d = NULL;
      if (cudaMalloc(&d, sizeof(uint16_t) * numel[p]) != cudaSuccess) return fail("cudaMalloc");
      cudaMemcpy(d, h, sizeof(uint16_t) * numel[p], cudaMemcpyHostToDevice);
      dg[k * P + p] = d;
      if (cudaMalloc((void**)&ds[k * P + p], sizeof(float) * shard_n[p]) != cudaSuccess) return fail("cudaMalloc");
    }
  uint16_t* hbuf = malloc(sizeof(uint16_t) * N * S);
  for (int64_t i = 0; i < N * S; ++i) hbuf[i] = value(9, 9, (uint32_t)i);
  uint16_t* dbuf = NULL;
  cudaMalloc((void**)&dbuf, sizeof(uint16_t) * N * S);
  cudaMemcpy(dbuf, hbuf, sizeof(uint16_t) * N * S, cudaMemcpyHostToDevice);
  for (int p = 0; p < P; ++p) cudaMalloc((void**)&dp[p], sizeof(uint16_t) * numel[p]);

  /* the two operations, on the default stream */
  if (tide_rs_bf16_to_fp32(lay, dg, ds, 0.25f, NULL) != TIDE_OK) return fail("tide_rs_bf16_to_fp32");
  if (tide_ag_place(lay, dbuf, dp, NULL) != TIDE_OK) return fail("tide_ag_place");
  if (cudaDeviceSynchronize() != cudaSuccess) return fail("cudaDeviceSynchronize");

  /* oracle results on the host */
  float* os[N * P];
  uint16_t* op[P];
  for (int i = 0; i < N * P; ++i) os[i] = malloc(sizeof(float) * shard_n[i % P]);
  for (int p = 0; p < P; ++p) op[p] = malloc(sizeof(uint16_t) * numel[p]);
  if (oracle_rs(N, P, d0, inner, (const uint16_t* const*)hg, os, 0.25f) != 0) return fail("oracle_rs refused");
  oracle_ag_place(N, P, d0, inner, offs, S, hbuf, op);

  long bad = 0, checked = 0;
  for (int i = 0; i < N * P; ++i) {
    float* got = malloc(sizeof(float) * shard_n[i % P]);
    cudaMemcpy(got, ds[i], sizeof(float) * shard_n[i % P], cudaMemcpyDeviceToHost);
    bad += memcmp(got, os[i], sizeof(float) * shard_n[i % P]) != 0;
    checked += shard_n[i % P];
    free(got);
  }
  for (int p = 0; p < P; ++p) {
    uint16_t* got = malloc(sizeof(uint16_t) * numel[p]);
    cudaMemcpy(got, dp[p], sizeof(uint16_t) * numel[p], cudaMemcpyDeviceToHost);
    bad += memcmp(got, op[p], sizeof(uint16_t) * numel[p]) != 0;
    checked += numel[p];
    free(got);
  }
  tide_layout_destroy(lay);
  if (bad) {
    fprintf(stderr, "FAIL: %ld output tensors differ from the oracle\n", bad);
    return 1;
  }
  printf("ok: %ld elements bit-exact against the oracle\n", checked);
  return 0;
}
