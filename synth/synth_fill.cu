// Device side of the synthetic input generator (see synth.h): fills device
// buffers in place so that multi-GB per-rank gradient sets never pass
// through host memory.  Built into libtide_synth.so, separate from the
// product library.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

__global__ void synth_fill_kernel(uint16_t* __restrict__ out, int64_t n, uint64_t key,
                                  uint64_t first, float amp, uint32_t outlier_every,
                                  float outlier_mult) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = synth_bf16(key, first + (uint64_t)i, amp, outlier_every, outlier_mult);
}

__global__ void synth_fill_f32_kernel(float* __restrict__ out, int64_t n, uint64_t key,
                                      uint64_t first, float amp) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = synth_f32(key, first + (uint64_t)i, amp);
}

__global__ void synth_set_u16_kernel(uint16_t* __restrict__ out, int64_t n, uint16_t v) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = v;
}

int grid_for(int64_t n) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

#define SYNTH_EXPORT __attribute__((visibility("default")))

extern "C" {

// out[i] = synth_bf16(key, first + i, ...) for i in [0, n), on `stream`.
// Returns the cudaError_t of the launch (0 on success).
SYNTH_EXPORT int synth_fill_bf16_device(uint16_t* out, int64_t n, uint64_t key, uint64_t first, float amp,
                           uint32_t outlier_every, float outlier_mult, void* stream) {
  if (n <= 0) return 0;
  synth_fill_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, key, first, amp,
                                                                  outlier_every, outlier_mult);
  return (int)cudaGetLastError();
}

// out[i] = synth_f32(key, first + i, amp) for i in [0, n), on `stream`.
SYNTH_EXPORT int synth_fill_f32_device(float* out, int64_t n, uint64_t key, uint64_t first, float amp,
                                       void* stream) {
  if (n <= 0) return 0;
  synth_fill_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, key, first, amp);
  return (int)cudaGetLastError();
}

// out[i] = v for i in [0, n): sentinel and guard-band fills.
SYNTH_EXPORT int synth_set_u16_device(uint16_t* out, int64_t n, uint16_t v, void* stream) {
  if (n <= 0) return 0;
  synth_set_u16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, v);
  return (int)cudaGetLastError();
}

}  // extern "C"
