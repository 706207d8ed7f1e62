/*
 * The no-allocation reduce-scatter across a device reset, from plain C.
 *
 * The library remembers which tables its fixed device array holds so that a
 * repeated call (same layout, stream and pointers) copies nothing.  A
 * cudaDeviceReset destroys the context: the array is loaded again (possibly
 * at another address) and its contents are gone, while a caller that
 * allocates again often gets the same addresses back.  The call after the
 * reset must notice the new context, look the array up again and copy.
 *
 * Values are small integers, so every sum is exact in fp32 in any order and
 * the expected shards follow in closed form:
 *   g[k][p][e] = (e mod 7) + k + base   =>   shard = scale * (N*((e mod 7) + base) + N(N-1)/2)
 * Prints "ok: ..." and exits 0 on success.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tide.h"

enum { N = 4, P = 2 };
static const int64_t D0[P] = {37, 10};
static const int64_t INNER[P] = {24, 1};

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s (%s)\n", what, tide_last_error());
  return 1;
}

static uint16_t bf16_of_small_int(int v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16); /* small integers are exact in bf16 */
}

static void* g_grad[N * P];
static void* g_shard[N * P];

static int alloc_and_fill(int base) {
  for (int k = 0; k < N; ++k)
    for (int p = 0; p < P; ++p) {
      const int64_t n = D0[p] * INNER[p];
      const int64_t c = (D0[p] + N - 1) / N;
      uint16_t* h = malloc(sizeof(uint16_t) * n);
      for (int64_t e = 0; e < n; ++e) h[e] = bf16_of_small_int((int)(e % 7) + k + base);
      if (cudaMalloc(&g_grad[k * P + p], sizeof(uint16_t) * n) != cudaSuccess) return fail("cudaMalloc");
      if (cudaMemcpy(g_grad[k * P + p], h, sizeof(uint16_t) * n, cudaMemcpyHostToDevice) != cudaSuccess)
        return fail("cudaMemcpy");
      free(h);
      if (cudaMalloc(&g_shard[k * P + p], sizeof(float) * c * INNER[p]) != cudaSuccess) return fail("cudaMalloc");
      if (cudaMemset(g_shard[k * P + p], 0xFF, sizeof(float) * c * INNER[p]) != cudaSuccess)
        return fail("cudaMemset");
    }
  return 0;
}

static int check(int base, float scale) {
  long bad = 0;
  for (int r = 0; r < N; ++r)
    for (int p = 0; p < P; ++p) {
      const int64_t c = (D0[p] + N - 1) / N;
      const int64_t n = c * INNER[p];
      float* h = malloc(sizeof(float) * n);
      if (cudaMemcpy(h, g_shard[r * P + p], sizeof(float) * n, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("cudaMemcpy back");
      for (int64_t e = 0; e < n; ++e) {
        const int64_t i = r * c * INNER[p] + e; /* element of the full gradient */
        const float want = i < D0[p] * INNER[p]
                               ? scale * (float)(N * ((int)(i % 7) + base) + N * (N - 1) / 2)
                               : 0.0f;
        bad += memcmp(&h[e], &want, sizeof want) != 0;
      }
      free(h);
    }
  return bad ? fail("shard mismatch") : 0;
}

int main(void) {
  int32_t ndims[P] = {2, 1};
  int64_t dims[3] = {D0[0], INNER[0], D0[1]};
  tide_layout_t lay = NULL;
  if (tide_layout_create(P, ndims, dims, N, &lay) != TIDE_OK) return fail("tide_layout_create");
  const float scale = 0.5f;

  if (alloc_and_fill(0)) return 1;
  void* first[N * P];
  memcpy(first, g_grad, sizeof first);
  if (tide_rs_bf16_to_fp32_noalloc(lay, (const uint16_t* const*)g_grad, (float* const*)g_shard, scale, NULL) !=
      TIDE_OK)
    return fail("no-allocation call before the reset");
  if (cudaDeviceSynchronize() != cudaSuccess) return fail("cudaDeviceSynchronize");
  if (check(0, scale)) return 1;

  if (cudaDeviceReset() != cudaSuccess) return fail("cudaDeviceReset");

  if (alloc_and_fill(3)) return 1;
  const int same = memcmp(first, g_grad, sizeof first) == 0;
  for (int call = 0; call < 2; ++call) { /* the second call repeats with nothing to copy */
    if (cudaMemset(g_shard[0], 0xFF, 4) != cudaSuccess) return fail("cudaMemset");
    if (tide_rs_bf16_to_fp32_noalloc(lay, (const uint16_t* const*)g_grad, (float* const*)g_shard, scale,
                                     NULL) != TIDE_OK)
      return fail("no-allocation call after the reset");
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("cudaDeviceSynchronize");
    if (check(3, scale)) return 1;
  }
  tide_layout_destroy(lay);
  printf("ok: results exact before and after cudaDeviceReset (allocations at the same addresses: %s)\n",
         same ? "yes" : "no");
  return 0;
}
