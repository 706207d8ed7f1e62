// HBM ceilings for the benchmark's roofline: streams with a fixed mix of
// reads and writes, shaped like the reduce-scatter (one CTA per tile, 16-byte
// streaming loads that skip L1, evict-first 16-byte stores, all of a
// thread's loads issued before any is used).
//
// The measured copy bandwidth the roofline divides by is a 1:1 copy.  The
// reduce-scatter reads 2N bytes for every 4 it writes (4:1 at N = 8, 8:1 at
// N = 16), and HBM reads and writes do not cost the same, so a kernel can
// stream above the 1:1 figure.  These streams measure what a read-only, a
// write-only and an R:1 read:write stream of the same shape reach on this
// GPU, so the reduce-scatter can be compared with a ceiling of its own mix.
// The few-CTA streams measure what one SM moves, the bound of the CTA-capped
// kernels.
//
// Used only by bench.py; not part of the library.
#include <cuda_runtime.h>
#include <stdint.h>

#define HBM_API __attribute__((visibility("default")))

namespace {

constexpr int kThreads = 512;
constexpr int kVecPerThread = 4;  // 16-byte vectors per thread per source
constexpr int64_t kTileVecs = (int64_t)kThreads * kVecPerThread;  // 32 KiB per source

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void xor_into(uint4& a, const uint4& b) {
  a.x ^= b.x;
  a.y ^= b.y;
  a.z ^= b.z;
  a.w ^= b.w;
}

// Read-only: every CTA streams one 64 KiB tile of `src` (8 loads in flight
// per thread); the XOR of what it read is stored only when it equals a value
// no input holds (so the loads stay).
constexpr int kReadVec = 8;
__global__ void __launch_bounds__(kThreads) read_kernel(const uint4* src, int64_t nvec, uint4* sink) {
  const int64_t base = (int64_t)blockIdx.x * kThreads * kReadVec;
  uint4 acc = make_uint4(0, 0, 0, 0);
  uint4 d[kReadVec];
#pragma unroll
  for (int u = 0; u < kReadVec; ++u) {
    const int64_t i = base + threadIdx.x + (int64_t)u * kThreads;
    d[u] = i < nvec ? ld_stream(src + i) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < kReadVec; ++u) xor_into(acc, d[u]);
  if (acc.x == 0x9E3779B9u && acc.y == 0x7F4A7C15u && acc.z == 0xF39CC060u && acc.w == 0x5CEDC834u)
    sink[0] = acc;
}

// Write-only: every CTA fills one tile of `dst`.
__global__ void __launch_bounds__(kThreads) write_kernel(uint4* dst, int64_t nvec, uint32_t v) {
  const int64_t base = (int64_t)blockIdx.x * kTileVecs;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int64_t i = base + threadIdx.x + (int64_t)u * kThreads;
    if (i < nvec) st_stream(dst + i, make_uint4(v, v ^ (uint32_t)i, v, (uint32_t)i));
  }
}

// R:1 read:write: output vector i is the XOR of vector i of R equally long
// source regions (src + k * nvec), as the reduce-scatter reads the same
// offset of N gradients for every result.  U output vectors per pass: all
// R * U loads of a pass are in flight before the XOR (8 loads per thread for
// R <= 8, as the reduce-scatter keeps 8 ranks' loads in flight).
template <int R, int U>
__global__ void __launch_bounds__(kThreads) mix_kernel(const uint4* src, uint4* dst, int64_t nvec) {
  static_assert(kVecPerThread % U == 0, "whole passes");
  const int64_t base = (int64_t)blockIdx.x * kTileVecs;
#pragma unroll 1
  for (int u0 = 0; u0 < kVecPerThread; u0 += U) {
    uint4 d[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + threadIdx.x + (int64_t)(u0 + u) * kThreads;
#pragma unroll
      for (int k = 0; k < R; ++k) d[u][k] = i < nvec ? ld_stream(src + (int64_t)k * nvec + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + threadIdx.x + (int64_t)(u0 + u) * kThreads;
      uint4 acc = d[u][0];
#pragma unroll
      for (int k = 1; k < R; ++k) xor_into(acc, d[u][k]);
      if (i < nvec) st_stream(dst + i, acc);
    }
  }
}

// Few-CTA streams, the shape of the CTA-capped kernels: `grid` CTAs of 1024
// threads loop over the buffer, every thread with 8 16-byte accesses in
// flight, so each CTA holds an SM and the rate per CTA is what one SM
// moves.  MODE 0 reads (XOR kept as in read_kernel), 1 writes, 2 copies.
constexpr int kSmThreads = 1024;
constexpr int kSmVec = 8;
template <int MODE>
__global__ void __launch_bounds__(kSmThreads, 1) sm_stream_kernel(const uint4* src, uint4* dst, int64_t nvec,
                                                                  uint4* sink) {
  constexpr int64_t kChunk = (int64_t)kSmThreads * kSmVec;
  uint4 acc = make_uint4(0, 0, 0, 0);
  for (int64_t base = (int64_t)blockIdx.x * kChunk; base < nvec; base += (int64_t)gridDim.x * kChunk) {
    if constexpr (MODE == 1) {
#pragma unroll
      for (int u = 0; u < kSmVec; ++u) {
        const int64_t i = base + threadIdx.x + (int64_t)u * kSmThreads;
        if (i < nvec) st_stream(dst + i, make_uint4((uint32_t)i, 1u, 2u, 3u));
      }
    } else {
      uint4 d[kSmVec];
#pragma unroll
      for (int u = 0; u < kSmVec; ++u) {
        const int64_t i = base + threadIdx.x + (int64_t)u * kSmThreads;
        d[u] = i < nvec ? ld_stream(src + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kSmVec; ++u) {
        const int64_t i = base + threadIdx.x + (int64_t)u * kSmThreads;
        if constexpr (MODE == 2) {
          if (i < nvec) st_stream(dst + i, d[u]);
        } else {
          xor_into(acc, d[u]);
        }
      }
    }
  }
  if (MODE == 0 && acc.x == 0x9E3779B9u && acc.y == 0x7F4A7C15u && acc.z == 0xF39CC060u && acc.w == 0x5CEDC834u)
    sink[0] = acc;
}

int grid_of(int64_t nvec) { return (int)((nvec + kTileVecs - 1) / kTileVecs); }

}  // namespace

extern "C" {

// Each call launches one kernel on `stream` and returns its cudaError_t.
// Sizes are in bytes, multiples of 16; pointers 16-byte aligned.
HBM_API int hbm_read(const void* src, int64_t bytes, void* sink16, cudaStream_t stream) {
  const int64_t nvec = bytes / 16;
  if (nvec <= 0) return 0;
  const int g = (int)((nvec + (int64_t)kThreads * kReadVec - 1) / ((int64_t)kThreads * kReadVec));
  read_kernel<<<g, kThreads, 0, stream>>>((const uint4*)src, nvec, (uint4*)sink16);
  return (int)cudaGetLastError();
}

HBM_API int hbm_write(void* dst, int64_t bytes, uint32_t value, cudaStream_t stream) {
  const int64_t nvec = bytes / 16;
  if (nvec <= 0) return 0;
  write_kernel<<<grid_of(nvec), kThreads, 0, stream>>>((uint4*)dst, nvec, value);
  return (int)cudaGetLastError();
}

// Reads `ratio` * out_bytes from src (ratio regions of out_bytes each) and
// writes out_bytes to dst; ratio is 1, 2, 4, 8 or 16.
HBM_API int hbm_mix(const void* src, void* dst, int64_t out_bytes, int ratio, cudaStream_t stream) {
  const int64_t nvec = out_bytes / 16;
  if (nvec <= 0) return 0;
  const uint4* s = (const uint4*)src;
  uint4* d = (uint4*)dst;
  const int g = grid_of(nvec);
  switch (ratio) {
    case 1: mix_kernel<1, 4><<<g, kThreads, 0, stream>>>(s, d, nvec); break;
    case 2: mix_kernel<2, 4><<<g, kThreads, 0, stream>>>(s, d, nvec); break;
    case 4: mix_kernel<4, 2><<<g, kThreads, 0, stream>>>(s, d, nvec); break;
    case 8: mix_kernel<8, 1><<<g, kThreads, 0, stream>>>(s, d, nvec); break;
    case 16: mix_kernel<16, 1><<<g, kThreads, 0, stream>>>(s, d, nvec); break;
    default: return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

// `grid` persistent 1024-thread CTAs streaming `bytes`: mode 0 reads src,
// 1 writes dst, 2 copies src to dst (bytes read and bytes written each).
HBM_API int hbm_sm_stream(const void* src, void* dst, int64_t bytes, int mode, int grid, void* sink16,
                          cudaStream_t stream) {
  const int64_t nvec = bytes / 16;
  if (nvec <= 0 || grid <= 0) return 0;
  const uint4* s = (const uint4*)src;
  uint4* d = (uint4*)dst;
  switch (mode) {
    case 0: sm_stream_kernel<0><<<grid, kSmThreads, 0, stream>>>(s, d, nvec, (uint4*)sink16); break;
    case 1: sm_stream_kernel<1><<<grid, kSmThreads, 0, stream>>>(s, d, nvec, (uint4*)sink16); break;
    case 2: sm_stream_kernel<2><<<grid, kSmThreads, 0, stream>>>(s, d, nvec, (uint4*)sink16); break;
    default: return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // extern "C"
