// Reduce-scatter math and all-gather placement kernels for sm_103a.
//
// Both are HBM-streaming kernels: the reduce-scatter reads N bf16 values and
// writes one fp32 value per element (about one fp32 add per 2 bytes read),
// the placement is a segmented bit copy.  Neither is a dense contraction, so
// there is no tensor-core path; what matters is 16-byte coalesced accesses,
// enough bytes in flight per SM and a flat tile list that balances many
// small tensors.
//
// Sources: "FSDP通信终局：TIDE零拷贝集合通信优化" §TIDE的设计思路 (TIDE-RS:
// per-parameter bf16 gradients reduced straight into fp32 shards; TIDE-AG:
// shards delivered straight into parameter storage; short-lived CTAs) and
// §FSDP2通信开销的根源 (rank-major buffers, reduce-scatter semantics).
#include <cuda_runtime.h>

#include <algorithm>
#include <stdint.h>

#include "tide_internal.h"

namespace tide {
namespace {

// ---------------------------------------------------------------- memory ops
// Streaming 16-byte load of data that is read exactly once: read-only path,
// no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
  uint16_t r;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// Streaming (evict-first) stores: outputs are not re-read by this kernel.
__device__ __forceinline__ void st_stream(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Plain 16-byte store / load (write-back, normal L2 priority).
__device__ __forceinline__ void st_plain(void* p, uint4 v) { *(uint4*)p = v; }
__device__ __forceinline__ uint4 ld_plain(const void* p) { return *(const uint4*)p; }

#ifndef TIDE_AG_STREAMING  // 1: the placement copy uses streaming stores and no-allocate loads
#define TIDE_AG_STREAMING 1
#endif

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// bf16 -> fp32 is exact: a bf16 is the upper half of an fp32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// acc[0..7] += the 8 bf16 values packed in v (in element order).
__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v) {
  acc[0] = __fadd_rn(acc[0], bf16_lo(v.x));
  acc[1] = __fadd_rn(acc[1], bf16_hi(v.x));
  acc[2] = __fadd_rn(acc[2], bf16_lo(v.y));
  acc[3] = __fadd_rn(acc[3], bf16_hi(v.y));
  acc[4] = __fadd_rn(acc[4], bf16_lo(v.z));
  acc[5] = __fadd_rn(acc[5], bf16_hi(v.z));
  acc[6] = __fadd_rn(acc[6], bf16_lo(v.w));
  acc[7] = __fadd_rn(acc[7], bf16_hi(v.w));
}

// Debug builds: false when the tile addresses anything outside the buffers of
// its call (tile_in_range); `reporter` then sets the range bit of the error
// word, and the caller skips the tile.  Release builds: always true.
__device__ __forceinline__ bool tile_ok(const Tile& t, int kind, const Extents& e, int* err, bool reporter) {
#if TIDE_DEBUG
  if (e.grad_numel && !tile_in_range(t, kind, e)) {
    if (reporter && err) atomicOr(err, kDevErrRange);
    return false;
  }
#else
  (void)t, (void)kind, (void)e, (void)err, (void)reporter;
#endif
  return true;
}

// ---------------------------------------------------------------- reduce-scatter
// One group of G ranks starting at rank k0: issue all G*V loads, then add
// them in ascending rank order.  FULL means k0 + G <= N is known.
// Vector u of a thread is vector v0 + u * stride of the run.
template <int G, int V, bool FULL>
__device__ __forceinline__ void rs_group(float (&acc)[V][8], const uint16_t* const* s_src, int k0,
                                         int n, int v0, int nvec, int stride) {
  uint4 d[G][V];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int u = 0; u < V; ++u)
      if ((FULL || k0 + j < n) && v0 + u * stride < nvec)
        d[j][u] = ld_stream(s_src[k0 + j] + 8 * (v0 + u * stride));
#pragma unroll
  for (int j = 0; j < G; ++j)
    if (FULL || k0 + j < n)
#pragma unroll
      for (int u = 0; u < V; ++u) add8(acc[u], d[j][u]);
}

// One tile = a run of `len` elements of parameter p that lands in rank r's
// shard.  Every rank k contributes the element at the same offset of its own
// gradient (the shard rows are the same rows in every rank's full gradient),
// so the tile reads N equally-long contiguous runs and writes one.
//
// Each thread owns V 8-element vectors per pass.  Loads are issued in
// groups of G ranks (all G*V 16-byte loads before any add) and the adds run
// in ascending rank order, so the fp32 result equals the sequential sum
// acc = ((0 + g_0) + g_1) + ... + g_{N-1}, then one multiply by the scale.
// NFIX > 0 fixes N at compile time (full unroll, no predicates).  The N
// source pointers of a tile are staged in shared memory, double-buffered so
// one barrier per tile suffices: a thread can only write buffer b again after
// every thread has passed the barrier of the tile in between.
template <int THREADS, int NFIX, int G, int V>
__global__ void __launch_bounds__(THREADS, TIDE_RS_MIN_BLOCKS) rs_kernel(RsArgs a) {
  extern __shared__ const uint16_t* s_src[];  // [2][N] source pointers
  const int N = NFIX > 0 ? NFIX : a.num_ranks;
  int buf = 0;
  for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, a.kind, a.ext, a.err, threadIdx.x == 0)) continue;  // uniform over the CTA
    float* __restrict__ out = a.stab[(int64_t)tile.r * a.num_params + tile.p] + tile.dst;

    if (tile.flags & kTileZero) {  // padding rows of the shard
      if (tile.flags & kTileVec) {
        const int nv = tile.len >> 2;
        for (int i = threadIdx.x; i < nv; i += THREADS) st_stream(out + 4 * i, 0.f, 0.f, 0.f, 0.f);
        for (int e = 4 * nv + threadIdx.x; e < tile.len; e += THREADS) out[e] = 0.f;
      } else {
        for (int e = threadIdx.x; e < tile.len; e += THREADS) out[e] = 0.f;
      }
      continue;
    }

    const uint16_t** sp = s_src + buf * N;
    buf ^= 1;
    for (int k = threadIdx.x; k < N; k += THREADS) sp[k] = a.gtab[(int64_t)tile.p * N + k] + tile.src;
    __syncthreads();

    if (tile.flags & kTileVec) {
      const int nvec = tile.len >> 3;
      for (int v0 = threadIdx.x; v0 < nvec; v0 += V * THREADS) {
        float acc[V][8];
#pragma unroll
        for (int u = 0; u < V; ++u)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
        if constexpr (NFIX > 0 && (THREADS <= 256 || NFIX <= G)) {
#pragma unroll
          for (int k0 = 0; k0 < NFIX; k0 += G) rs_group<G, V, true>(acc, sp, k0, N, v0, nvec, THREADS);
        } else if constexpr (NFIX > 0) {
          // fat CTAs: one group of loads in flight per thread, no spills
#pragma unroll 1
          for (int k0 = 0; k0 < NFIX; k0 += G) rs_group<G, V, true>(acc, sp, k0, N, v0, nvec, THREADS);
        } else {
          for (int k0 = 0; k0 < N; k0 += G) rs_group<G, V, false>(acc, sp, k0, N, v0, nvec, THREADS);
        }
#pragma unroll
        for (int u = 0; u < V; ++u) {
          const int v = v0 + u * THREADS;
          if (v < nvec) {
            float* o = out + 8 * v;
            st_stream(o, __fmul_rn(acc[u][0], a.scale), __fmul_rn(acc[u][1], a.scale),
                      __fmul_rn(acc[u][2], a.scale), __fmul_rn(acc[u][3], a.scale));
            st_stream(o + 4, __fmul_rn(acc[u][4], a.scale), __fmul_rn(acc[u][5], a.scale),
                      __fmul_rn(acc[u][6], a.scale), __fmul_rn(acc[u][7], a.scale));
          }
        }
      }
      for (int e = 8 * nvec + threadIdx.x; e < tile.len; e += THREADS) {
        float acc = 0.f;
        for (int k = 0; k < N; ++k) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(sp[k] + e)));
        out[e] = __fmul_rn(acc, a.scale);
      }
    } else {  // a run whose source is not 16-byte aligned: element by element
      for (int e = threadIdx.x; e < tile.len; e += THREADS) {
        float acc = 0.f;
        for (int k = 0; k < N; ++k) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(sp[k] + e)));
        out[e] = __fmul_rn(acc, a.scale);
      }
    }
  }
}

// CTA-capped form: every warp of the (few, fat) CTAs walks its own tiles —
// tile t goes to warp t mod (warps in the grid) — with its N source pointers
// in its own shared-memory slot, so no CTA-wide barrier ties the warps
// together.  In the CTA-wide loop above, all of a fat CTA's warps issue
// their loads, wait and add in step, and an SM holding one streams about
// half of what its loads in flight allow; here, while some warps add, the
// others' loads are in flight.  Same sums in the same order: each lane owns
// whole 8-element vectors, strided by the warp width.  NFIX > 0 fixes N;
// NFIX == 0 takes N at run time (N <= kRsWarpMaxRanks).
template <int THREADS, int NFIX, int G, int V>
__global__ void __launch_bounds__(THREADS, 1) rs_warp_kernel(RsArgs a) {
  extern __shared__ const uint16_t* s_src[];  // [THREADS / 32][N] source pointers
  const int N = NFIX > 0 ? NFIX : a.num_ranks;
  const int lane = (int)threadIdx.x & 31, warp = (int)threadIdx.x >> 5;
  const uint16_t** sp = s_src + warp * N;
  constexpr int kWarps = THREADS / 32;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < a.num_tiles; t += (int64_t)gridDim.x * kWarps) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, a.kind, a.ext, a.err, lane == 0)) continue;  // uniform over the warp
    float* __restrict__ out = a.stab[(int64_t)tile.r * a.num_params + tile.p] + tile.dst;

    if (tile.flags & kTileZero) {  // padding rows of the shard
      if (tile.flags & kTileVec) {
        const int nv = tile.len >> 2;
        for (int i = lane; i < nv; i += 32) st_stream(out + 4 * i, 0.f, 0.f, 0.f, 0.f);
        for (int e = 4 * nv + lane; e < tile.len; e += 32) out[e] = 0.f;
      } else {
        for (int e = lane; e < tile.len; e += 32) out[e] = 0.f;
      }
      continue;
    }

    __syncwarp();  // every lane is done with the previous tile's pointers
    for (int k = lane; k < N; k += 32) sp[k] = a.gtab[(int64_t)tile.p * N + k] + tile.src;
    __syncwarp();

    if (tile.flags & kTileVec) {
      const int nvec = tile.len >> 3;
      for (int v0 = lane; v0 < nvec; v0 += V * 32) {
        float acc[V][8];
#pragma unroll
        for (int u = 0; u < V; ++u)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
        if constexpr (NFIX > 0) {
#pragma unroll 1
          for (int k0 = 0; k0 < NFIX; k0 += G) rs_group<G, V, true>(acc, sp, k0, N, v0, nvec, 32);
        } else {
          for (int k0 = 0; k0 < N; k0 += G) rs_group<G, V, false>(acc, sp, k0, N, v0, nvec, 32);
        }
#pragma unroll
        for (int u = 0; u < V; ++u) {
          const int v = v0 + u * 32;
          if (v < nvec) {
            float* o = out + 8 * v;
            st_stream(o, __fmul_rn(acc[u][0], a.scale), __fmul_rn(acc[u][1], a.scale),
                      __fmul_rn(acc[u][2], a.scale), __fmul_rn(acc[u][3], a.scale));
            st_stream(o + 4, __fmul_rn(acc[u][4], a.scale), __fmul_rn(acc[u][5], a.scale),
                      __fmul_rn(acc[u][6], a.scale), __fmul_rn(acc[u][7], a.scale));
          }
        }
      }
      for (int e = 8 * nvec + lane; e < tile.len; e += 32) {
        float acc = 0.f;
        for (int k = 0; k < N; ++k) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(sp[k] + e)));
        out[e] = __fmul_rn(acc, a.scale);
      }
    } else {  // a run whose source is not 16-byte aligned: element by element
      for (int e = lane; e < tile.len; e += 32) {
        float acc = 0.f;
        for (int k = 0; k < N; ++k) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(sp[k] + e)));
        out[e] = __fmul_rn(acc, a.scale);
      }
    }
  }
}

// ---------------------------------------------------------------- placement
// One tile = a contiguous run of rank r's chunk of parameter p: a copy from
// gathered[r*S + o_p + ...] to params[p][r*c_p*inner_p + ...].  U 16-byte
// vectors per thread are loaded before any is stored.  TO_BUF runs the same
// copy backwards (Slot-Reuse staging of a gradient into the rank-major slot).
// A CTA is WORKERS independent groups of THREADS / WORKERS threads, each
// walking its own tiles: one group per CTA over every SM; in capped mode one
// per warp in small grids (small_fat_grid), else two 512-thread groups.
template <int THREADS, int WORKERS, int U, bool TO_BUF>
__global__ void __launch_bounds__(THREADS) ag_kernel(AgArgs a) {
  constexpr int WT = THREADS / WORKERS;
  static_assert(THREADS % WORKERS == 0 && WT % 32 == 0, "workers are whole warps");
  const int lane = (int)threadIdx.x % WT;
  for (int64_t t = (int64_t)blockIdx.x * WORKERS + (int)threadIdx.x / WT; t < a.num_tiles;
       t += (int64_t)gridDim.x * WORKERS) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, kKindCopy, a.ext, a.err, lane == 0)) continue;  // uniform over the group
    const uint16_t* __restrict__ src;
    uint16_t* __restrict__ dst;
    if constexpr (TO_BUF) {
      src = a.ptab[tile.p] + tile.dst;
      dst = const_cast<uint16_t*>(a.buf) + tile.src;
    } else {
      src = (a.bufs ? a.bufs[tile.r] : a.buf) + tile.src;
      dst = a.ptab[tile.p] + tile.dst;
    }
    if (tile.flags & kTileVec) {
      const int nvec = tile.len >> 3;
      for (int v0 = lane; v0 < nvec; v0 += U * WT) {
        uint4 d[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * WT < nvec)
            d[u] = TIDE_AG_STREAMING ? ld_stream(src + 8 * (v0 + u * WT))
                                     : ld_plain(src + 8 * (v0 + u * WT));
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * WT < nvec) {
            if (TIDE_AG_STREAMING)
              st_stream(dst + 8 * (v0 + u * WT), d[u]);
            else
              st_plain(dst + 8 * (v0 + u * WT), d[u]);
          }
      }
      for (int e = 8 * nvec + lane; e < tile.len; e += WT) dst[e] = ld_stream_u16(src + e);
    } else {
      for (int e = lane; e < tile.len; e += WT) dst[e] = ld_stream_u16(src + e);
    }
  }
}

// ---------------------------------------------------------------- bulk-copy placement
// The same segmented copy driven by the TMA engine: one lane per CTA issues
// cp.async.bulk global->shared copies of TIDE_BULK_CHUNK bytes into a ring of
// stages (completion tracked by one mbarrier per stage) and
// cp.async.bulk shared->global copies out of them, so the SM's load/store
// units carry almost nothing.  Only 16-byte-aligned vector runs go through
// the bulk path (their addresses and sizes are multiples of 16 bytes by
// construction); the rest of the warp copies unaligned runs and the < 8
// element tails with plain loads.  Every mbarrier wait is bounded by
// %globaltimer: on timeout the kernel sets *err, waits (bounded) for its own
// copies in flight and returns.
namespace bulk {

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// True once the phase with `parity` has completed; false after timeout_ns.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!mbar_test(bar, parity)) {
    if (now_ns() - t0 > timeout_ns) return false;
    __nanosleep(32);
  }
  return true;
}

// L2 policy for data touched once: evict first (as the streaming loads and
// stores of the load/store kernels).
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void g2s(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar,
                                    uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(saddr(smem)),
      "l"(gmem), "r"(bytes), "r"(saddr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void s2g(void* gmem, const void* smem, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gmem),
               "r"(saddr(smem)), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the `n` most recent bulk groups have finished reading shared memory.
template <int n>
__device__ __forceinline__ void wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(n) : "memory");
}

__device__ __forceinline__ void wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Walks this CTA's vector runs (tiles blockIdx.x, +gridDim.x, ...) in
// chunks of at most TIDE_BULK_CHUNK bytes.
struct Cursor {
  int64_t t;
  const unsigned char* src;
  unsigned char* dst;
  uint64_t bytes, off;
};

template <bool TO_BUF>
__device__ __forceinline__ bool next_chunk(Cursor& c, const AgArgs& a, const void*& src, void*& dst,
                                           uint32_t& n) {
  while (c.off >= c.bytes) {
    c.t += gridDim.x;
    if (c.t >= a.num_tiles) return false;
    const Tile tile = a.tiles[c.t];
    c.off = 0;
    if (!tile_ok(tile, kKindCopy, a.ext, nullptr, false)) {  // reported by the plain-copy pass
      c.bytes = 0;
      continue;
    }
    c.bytes = (tile.flags & kTileVec) ? (uint64_t)(tile.len & ~7) * 2u : 0u;
    const unsigned char* b = (const unsigned char*)(a.buf + tile.src);
    const unsigned char* q = (const unsigned char*)(a.ptab[tile.p] + tile.dst);
    c.src = TO_BUF ? q : b;
    c.dst = (unsigned char*)(TO_BUF ? b : q);
  }
  const uint64_t left = c.bytes - c.off;
  n = left < (uint64_t)TIDE_BULK_CHUNK ? (uint32_t)left : (uint32_t)TIDE_BULK_CHUNK;
  src = c.src + c.off;
  dst = c.dst + c.off;
  c.off += n;
  return true;
}

}  // namespace bulk

__device__ __forceinline__ uint64_t evict_first_policy_rs() { return bulk::evict_first_policy(); }

template <bool TO_BUF>
__global__ void __launch_bounds__(32) ag_bulk_kernel(AgArgs a) {
  constexpr int S = TIDE_BULK_STAGES;
  extern __shared__ __align__(128) unsigned char bulk_smem[];
  unsigned char(*stage)[TIDE_BULK_CHUNK] = (unsigned char(*)[TIDE_BULK_CHUNK])bulk_smem;
  uint64_t* full = (uint64_t*)(bulk_smem + (size_t)S * TIDE_BULK_CHUNK);  // S + 1; [S]: test hook

  // plain-copy parts: unaligned runs, and the < 8 element tails of vector runs
  for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, kKindCopy, a.ext, a.err, threadIdx.x == 0)) continue;
    const uint16_t* b = a.buf + tile.src;
    uint16_t* q = a.ptab[tile.p] + tile.dst;
    const uint16_t* src = TO_BUF ? q : b;
    uint16_t* dst = TO_BUF ? const_cast<uint16_t*>(b) : q;
    for (int e = ((tile.flags & kTileVec) ? (tile.len & ~7) : 0) + threadIdx.x; e < tile.len; e += 32)
      dst[e] = ld_stream_u16(src + e);
  }
  if (threadIdx.x != 0) return;

  for (int s = 0; s <= S; ++s) bulk::mbar_init(&full[s], 1);
  bulk::fence_mbar_init();
  if (a.test_stall_ns) {  // a barrier nothing arrives on: the wait must run out
    if (!bulk::mbar_wait(&full[S], 0, a.test_stall_ns)) atomicOr(a.err, kDevErrTimeout);
    return;
  }

  const uint64_t pol = bulk::evict_first_policy();
  bulk::Cursor lc{(int64_t)blockIdx.x - (int64_t)gridDim.x, nullptr, nullptr, 0, 0};
  bulk::Cursor sc = lc;
  const void* src;
  void* dst;
  uint32_t n;
  int64_t issued = 0;
  for (; issued < S - 1 && bulk::next_chunk<TO_BUF>(lc, a, src, dst, n); ++issued) {
    bulk::mbar_expect_tx(&full[issued % S], n);
    bulk::g2s(stage[issued % S], src, n, &full[issued % S], pol);
  }
  for (int64_t j = 0; j < issued; ++j) {
    const int s = (int)(j % S);
    if (!bulk::mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.timeout_ns)) {
      atomicOr(a.err, kDevErrTimeout);
      for (int64_t k = j; k < issued; ++k)  // loads that may still land in this CTA's shared memory
        bulk::mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.timeout_ns);
      bulk::wait_all();
      return;
    }
    bulk::next_chunk<TO_BUF>(sc, a, src, dst, n);
    bulk::s2g(dst, stage[s], n, pol);
    bulk::commit();
    // chunk `issued` goes to stage (j - 1) % S, last read by the store of
    // chunk j - 1: wait until only the store just issued may still read
    if (bulk::next_chunk<TO_BUF>(lc, a, src, dst, n)) {
      bulk::wait_read<1>();
      const int s2 = (int)(issued % S);
      bulk::mbar_expect_tx(&full[s2], n);
      bulk::g2s(stage[s2], src, n, &full[s2], pol);
      ++issued;
    }
  }
  bulk::wait_all();
}

// ---------------------------------------------------------------- bulk-staged reduce-scatter
// The reduce-scatter with its rank slices staged in shared memory by the TMA
// engine.  Warp 0 is the producer: per chunk of E elements of a vector run it
// issues N cp.async.bulk copies (one per rank, E*2 bytes each, spread over
// its lanes) into one stage of a ring and one expect-tx on that stage's
// "full" mbarrier.  Warps 1..8 consume: wait for "full", sum the N slices in
// ascending rank order from shared memory (__fadd_rn, the same sequence as
// the load/store kernel), write the fp32 results with streaming stores, and
// release the stage on its "empty" mbarrier.  The bulk-copy engine keeps
// ~192 KiB of slices in flight per SM with a seventh of the load/store
// kernel's warps resident (measured on GB300: 0.96-0.97 of its bandwidth
// over every SM, and per SM in a capped run 80 GB/s against the per-warp
// tile kernel's 110: there the SM's path out to L2 is the limit, not bytes
// in flight).  Zero tiles, unaligned runs and the
// < 8 element tails of vector runs are done by the consumers with plain
// loads.  Every wait is bounded as in the bulk-copy placement.
namespace bulk {

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}


}  // namespace bulk

constexpr int kRsBulkConsumerWarps = kRsBulkThreads / 32 - 1;
constexpr int kRsBulkConsumers = kRsBulkConsumerWarps * 32;
constexpr size_t kRsBulkRing = 196608;  // bytes of staged slices per CTA
constexpr int kRsBulkMaxStages = 32;

__device__ __forceinline__ void rs_scalar_run(const RsArgs& a, const Tile& tile, float* out, int e0,
                                              int tid, int nthreads) {
  const int N = a.num_ranks;
  const uint16_t* const* g = a.gtab + (int64_t)tile.p * N;
  for (int e = e0 + tid; e < tile.len; e += nthreads) {
    float acc = 0.f;
    for (int k = 0; k < N; ++k) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(g[k] + tile.src + e)));
    out[e] = __fmul_rn(acc, a.scale);
  }
}

// Ring geometry of the TMA-staged reduce-scatter, shared by the launcher and
// the kernel.  A stage holds the slices of G ranks (G = N: one stage per
// chunk; G < N: rank-group staging, a chunk spans `groups` consecutive
// stages), each slice E elements (a multiple of 8, so every copy is a
// multiple of 16 bytes).
struct RsBulkGeom {
  int G, groups, E;
  uint32_t slice, stage;
  int S;
};

__device__ __host__ __forceinline__ RsBulkGeom rs_bulk_geom(int n, int stage_target, int rank_group) {
  RsBulkGeom g;
  g.G = (rank_group > 0 && rank_group < n) ? rank_group : n;
  g.groups = (n + g.G - 1) / g.G;
  g.E = (stage_target / 2 / g.G) & ~7;
  g.slice = (uint32_t)g.E * 2u;
  g.stage = g.slice * (uint32_t)g.G;
  const size_t fit = g.stage ? kRsBulkRing / g.stage : 0;
  g.S = (int)(fit < (size_t)kRsBulkMaxStages ? fit : (size_t)kRsBulkMaxStages);
  return g;
}

// Rank-group staging keeps every consumer thread's partial sums of a chunk
// in registers across the chunk's stages: at most this many 8-element
// vectors per thread (a slice of up to 8 KiB).
constexpr int kRsBulkGroupVecs = 2;

__global__ void __launch_bounds__(kRsBulkThreads, 1) rs_bulk_kernel(RsArgs a) {
  extern __shared__ __align__(128) unsigned char rs_smem[];
  const int N = a.num_ranks;
  const RsBulkGeom geo = rs_bulk_geom(N, a.stage_bytes, a.rank_group);
  const int E = geo.E, S = geo.S, G = geo.G, groups = geo.groups;
  const uint32_t slice = geo.slice, stage_bytes = geo.stage;
  uint64_t* full = (uint64_t*)(rs_smem + (size_t)S * stage_bytes);
  uint64_t* empty = full + S;
  const uint16_t** ptrs = (const uint16_t**)(empty + S);  // producer's current sources
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      bulk::mbar_init(&full[s], 1);
      bulk::mbar_init(&empty[s], kRsBulkConsumerWarps);
    }
    bulk::fence_mbar_init();
  }
  __syncthreads();

  if (a.test_stall_ns) {  // wait on a phase nothing completes: must run out
    if (threadIdx.x == 0 && !bulk::mbar_wait(&full[0], 0, a.test_stall_ns)) atomicOr(a.err, kDevErrTimeout);
    return;
  }

  if (warp == 0) {  // ---------------- producer
    const uint64_t pol = evict_first_policy_rs();
    int64_t j = 0;  // stages issued
    for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
      const Tile tile = a.tiles[t];
      if (!tile_ok(tile, a.kind, a.ext, a.err, false)) continue;  // the consumers report it
      if ((tile.flags & kTileZero) || !(tile.flags & kTileVec)) continue;
      const int vec = tile.len & ~7;
      if (vec == 0) continue;
      __syncwarp();
      for (int k = lane; k < N; k += 32) ptrs[k] = a.gtab[(int64_t)tile.p * N + k] + tile.src;
      __syncwarp();
      for (int off = 0; off < vec; off += E) {
        const int n = min(E, vec - off);
        for (int g = 0; g < groups; ++g, ++j) {  // the chunk's rank groups, in rank order
          const int k0 = g * G, gk = min(G, N - k0);
          const int s = (int)(j % S);
          if (j >= S) {  // the consumers released this stage's previous contents
            int ok = lane == 0 ? (int)bulk::mbar_wait(&empty[s], (uint32_t)(((j / S) + 1) & 1), a.timeout_ns) : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
              if (lane == 0) atomicOr(a.err, kDevErrTimeout);
              // loads issued into the ring may still land: wait (bounded) for them
              for (int64_t k = (j >= S ? j - S : 0); k < j; ++k)
                if (lane == 0) bulk::mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.timeout_ns);
              return;
            }
          }
          if (lane == 0) bulk::mbar_expect_tx(&full[s], (uint32_t)gk * (uint32_t)n * 2u);
          __syncwarp();
          unsigned char* st = rs_smem + (size_t)s * stage_bytes;
          for (int k = lane; k < gk; k += 32)
            bulk::g2s(st + (size_t)k * slice, ptrs[k0 + k] + off, (uint32_t)n * 2u, &full[s], pol);
        }
      }
    }
    return;
  }

  // ---------------- consumers
  const int cid = threadIdx.x - 32;
  int64_t j = 0;  // stages consumed
  for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, a.kind, a.ext, a.err, cid == 0)) continue;  // the producer skips it too
    float* __restrict__ out = a.stab[(int64_t)tile.r * a.num_params + tile.p] + tile.dst;
    if (tile.flags & kTileZero) {
      for (int e = cid; e < tile.len; e += kRsBulkConsumers) out[e] = 0.f;
      continue;
    }
    if (!(tile.flags & kTileVec)) {
      rs_scalar_run(a, tile, out, 0, cid, kRsBulkConsumers);
      continue;
    }
    const int vec = tile.len & ~7;
    for (int off = 0; off < vec; off += E) {
      const int nv = min(E, vec - off) >> 3;
      if (groups == 1) {  // one stage holds every rank's slice of the chunk
        const int s = (int)(j % S);
        if (!bulk::mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.timeout_ns)) {
          atomicOr(a.err, kDevErrTimeout);
          return;
        }
        const unsigned char* st = rs_smem + (size_t)s * stage_bytes;
        for (int v = cid; v < nv; v += kRsBulkConsumers) {
          float acc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.f;
          for (int k = 0; k < N; ++k) add8(acc, *(const uint4*)(st + (size_t)k * slice + 16 * v));
          float* o = out + off + 8 * v;
          st_stream(o, __fmul_rn(acc[0], a.scale), __fmul_rn(acc[1], a.scale), __fmul_rn(acc[2], a.scale),
                    __fmul_rn(acc[3], a.scale));
          st_stream(o + 4, __fmul_rn(acc[4], a.scale), __fmul_rn(acc[5], a.scale), __fmul_rn(acc[6], a.scale),
                    __fmul_rn(acc[7], a.scale));
        }
        __syncwarp();
        if (lane == 0) bulk::mbar_arrive(&empty[s]);
        ++j;
        continue;
      }
      // rank-group staging: the chunk's groups arrive in consecutive stages;
      // each thread's vectors keep their sums in registers across them
      float acc[kRsBulkGroupVecs][8];
#pragma unroll
      for (int u = 0; u < kRsBulkGroupVecs; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
      for (int g = 0; g < groups; ++g, ++j) {
        const int s = (int)(j % S);
        if (!bulk::mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.timeout_ns)) {
          atomicOr(a.err, kDevErrTimeout);
          return;
        }
        const int gk = min(G, N - g * G);
        const unsigned char* st = rs_smem + (size_t)s * stage_bytes;
#pragma unroll
        for (int u = 0; u < kRsBulkGroupVecs; ++u) {
          const int v = cid + u * kRsBulkConsumers;
          if (v < nv)
            for (int k = 0; k < gk; ++k) add8(acc[u], *(const uint4*)(st + (size_t)k * slice + 16 * v));
        }
        __syncwarp();
        if (lane == 0) bulk::mbar_arrive(&empty[s]);
      }
#pragma unroll
      for (int u = 0; u < kRsBulkGroupVecs; ++u) {
        const int v = cid + u * kRsBulkConsumers;
        if (v < nv) {
          float* o = out + off + 8 * v;
          st_stream(o, __fmul_rn(acc[u][0], a.scale), __fmul_rn(acc[u][1], a.scale),
                    __fmul_rn(acc[u][2], a.scale), __fmul_rn(acc[u][3], a.scale));
          st_stream(o + 4, __fmul_rn(acc[u][4], a.scale), __fmul_rn(acc[u][5], a.scale),
                    __fmul_rn(acc[u][6], a.scale), __fmul_rn(acc[u][7], a.scale));
        }
      }
    }
    rs_scalar_run(a, tile, out, vec, cid, kRsBulkConsumers);  // < 8 element tail
  }
}

// ---------------------------------------------------------------- all-gather input pack
// fp32 -> bf16 bits, IEEE 754-2008 roundTiesToEven (§4.3.1) applied to the
// 16 dropped bits.  Adding 0x7FFF plus the lowest kept bit carries into the
// kept bits exactly when the dropped part is above half a bf16 ulp, or equal
// to it with an odd kept part; a carry out of the mantissa steps the
// exponent, which rounds the largest finite values up to infinity as the
// rule requires.  A NaN keeps its sign and top payload and is made quiet.
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (u >> 16) | 0x0040u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// One tile = a run of rank r's fp32 shard of parameter p, cast to bf16 into
// its slot gathered[r*S + o_p + ...].  Per 8 elements: two 16-byte loads,
// one 16-byte store; each thread loads U such vectors before it stores any.
// WORKERS as in ag_kernel.
template <int THREADS, int WORKERS, int U>
__global__ void __launch_bounds__(THREADS) pack_kernel(PackArgs a) {
  constexpr int WT = THREADS / WORKERS;
  static_assert(THREADS % WORKERS == 0 && WT % 32 == 0, "workers are whole warps");
  const int lane = (int)threadIdx.x % WT;
  for (int64_t t = (int64_t)blockIdx.x * WORKERS + (int)threadIdx.x / WT; t < a.num_tiles;
       t += (int64_t)gridDim.x * WORKERS) {
    const Tile tile = a.tiles[t];
    if (!tile_ok(tile, kKindPack, a.ext, a.err, lane == 0)) continue;  // uniform over the group
    const float* __restrict__ src = a.stab[(int64_t)tile.r * a.num_params + tile.p] + tile.src;
    uint16_t* __restrict__ dst = a.buf + tile.dst;
    int e0 = 0;
    if (tile.flags & kTileVec) {
      const int nvec = tile.len >> 3;
      for (int v0 = lane; v0 < nvec; v0 += U * WT) {
        uint4 x[U], y[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * WT < nvec) {
            x[u] = ld_stream(src + 8 * (v0 + u * WT));
            y[u] = ld_stream(src + 8 * (v0 + u * WT) + 4);
          }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * WT < nvec) {
            uint4 o;
            o.x = pack2(__uint_as_float(x[u].x), __uint_as_float(x[u].y));
            o.y = pack2(__uint_as_float(x[u].z), __uint_as_float(x[u].w));
            o.z = pack2(__uint_as_float(y[u].x), __uint_as_float(y[u].y));
            o.w = pack2(__uint_as_float(y[u].z), __uint_as_float(y[u].w));
            st_stream(dst + 8 * (v0 + u * WT), o);
          }
      }
      e0 = 8 * nvec;
    }
    for (int e = e0 + lane; e < tile.len; e += WT)
      dst[e] = (uint16_t)f32_to_bf16_bits(src[e]);
  }
}

// ---------------------------------------------------------------- dispatch
using RsKernel = void (*)(RsArgs);
using AgKernel = void (*)(AgArgs);

template <int T>
RsKernel rs_kernel_for(int32_t n) {
  switch (n) {
    case 1: return rs_kernel<T, 1, 1, 8>;
    case 2: return rs_kernel<T, 2, 2, 4>;
    case 3: return rs_kernel<T, 3, 3, 2>;
    case 4: return rs_kernel<T, 4, 4, 2>;
    case 5: return rs_kernel<T, 5, 5, 1>;
    case 6: return rs_kernel<T, 6, 6, 1>;
    case 7: return rs_kernel<T, 7, 7, 1>;
    case 8: return rs_kernel<T, 8, 8, 1>;
    case 16: return rs_kernel<T, 16, 8, 1>;
    case 32: return rs_kernel<T, 32, 8, 1>;
    // 16 loads in flight per thread at N = 64 (8 in fat CTAs, whose register
    // budget is 64): +4% on GB300; at N = 32 groups of 16 were slower
    case 64: return rs_kernel<T, 64, (T > 512 ? 8 : 16), 1>;
    default: return rs_kernel<T, 0, 8, 1>;
  }
}

RsKernel rs_kernel_for(int32_t n, bool fat) {
  return fat ? rs_kernel_for<kFatThreads>(n) : rs_kernel_for<kRsThreads>(n);
}

// Capped-mode kernels with per-warp tiles (N <= kRsWarpMaxRanks): the same
// loads in flight per thread as the fat CTA-wide kernels.
template <int T>
RsKernel rs_warp_kernel_for(int32_t n) {
  switch (n) {
    case 1: return rs_warp_kernel<T, 1, 1, 8>;
    case 2: return rs_warp_kernel<T, 2, 2, 4>;
    case 3: return rs_warp_kernel<T, 3, 3, 2>;
    case 4: return rs_warp_kernel<T, 4, 4, 2>;
    case 5: return rs_warp_kernel<T, 5, 5, 1>;
    case 6: return rs_warp_kernel<T, 6, 6, 1>;
    case 7: return rs_warp_kernel<T, 7, 7, 1>;
    case 8: return rs_warp_kernel<T, 8, 8, 1>;
    case 16: return rs_warp_kernel<T, 16, 8, 1>;
    case 32: return rs_warp_kernel<T, 32, 8, 1>;
    case 64: return rs_warp_kernel<T, 64, 8, 1>;
    default: return rs_warp_kernel<T, 0, 8, 1>;
  }
}

// Per-warp tiles for small capped grids.  Measured on GB300 (70B layer,
// N = 8): 1.24-1.28x the CTA-wide loop at 8-64 CTAs, level at 96, 0.92x at
// 152, where the kernel is bound by HBM rather than by each SM and the
// CTA-wide loop's longer runs per rank stream better.
bool rs_uses_warp_tiles(int32_t n, bool fat, int grid, int sms) {
  return n <= kRsWarpMaxRanks && small_fat_grid(fat, grid, sms);
}

// capped-mode CTAs: kFatThreads threads as TIDE_FAT_WORKERS independent groups
#ifndef TIDE_FAT_WORKERS
#define TIDE_FAT_WORKERS (TIDE_FAT_THREADS / TIDE_AG_THREADS)
#endif
constexpr int kFatWorkers = TIDE_FAT_WORKERS;
static_assert(kFatThreads % kFatWorkers == 0 && (kFatThreads / kFatWorkers) % 32 == 0,
              "a fat CTA is whole groups of whole warps");

// Small capped grids (small_fat_grid): every warp of a fat CTA is a group.
constexpr int kFatWarpWorkers = kFatThreads / 32;

template <bool TO_BUF>
AgKernel ag_kernel_for(bool fat, bool warps) {
  if (!fat) return ag_kernel<kAgThreads, 1, TIDE_AG_UNROLL, TO_BUF>;
  return warps ? ag_kernel<kFatThreads, kFatWarpWorkers, TIDE_AG_FAT_UNROLL, TO_BUF>
               : ag_kernel<kFatThreads, kFatWorkers, TIDE_AG_FAT_UNROLL, TO_BUF>;
}

}  // namespace

size_t rs_smem_bytes(int32_t num_ranks) { return 2 * sizeof(const uint16_t*) * (size_t)num_ranks; }

int rs_block(bool fat) { return fat ? kFatThreads : kRsThreads; }
int ag_block(bool fat) { return fat ? kFatThreads : kAgThreads; }

cudaError_t launch_rs(const RsArgs& a, int grid, bool fat, int sms, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  if (rs_uses_warp_tiles(a.num_ranks, fat, grid, sms)) {
    const size_t smem = sizeof(const uint16_t*) * (size_t)(kFatThreads / 32) * (size_t)a.num_ranks;
    rs_warp_kernel_for<kFatThreads>(a.num_ranks)<<<grid, kFatThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  const RsKernel k = rs_kernel_for(a.num_ranks, fat);
  const size_t smem = rs_smem_bytes(a.num_ranks);
  if (smem > 48 * 1024) {  // 2*N staged pointers: above 3072 ranks they need the opt-in size
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k<<<grid, rs_block(fat), smem, stream>>>(a);
  return cudaGetLastError();
}

// Placement and staging: in small capped grids one group per warp — measured
// on GB300 (70B / MoE layers) 1.02x the two 512-thread groups at 8-32 CTAs,
// 1.11-1.12x at 64, 0.96x at 152.
cudaError_t launch_ag(const AgArgs& a, int grid, bool fat, int sms, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  ag_kernel_for<false>(fat, small_fat_grid(fat, grid, sms))<<<grid, ag_block(fat), 0, stream>>>(a);
  return cudaGetLastError();
}

int pk_block(bool fat) { return fat ? kFatThreads : kAgThreads; }

cudaError_t launch_stage(const AgArgs& a, int grid, bool fat, int sms, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  ag_kernel_for<true>(fat, small_fat_grid(fat, grid, sms))<<<grid, ag_block(fat), 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_pack(const PackArgs& a, int grid, bool fat, int sms, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  if (small_fat_grid(fat, grid, sms))
    pack_kernel<kFatThreads, kFatWarpWorkers, TIDE_PACK_FAT_UNROLL><<<grid, kFatThreads, 0, stream>>>(a);
  else if (fat)
    pack_kernel<kFatThreads, kFatWorkers, TIDE_PACK_FAT_UNROLL><<<grid, kFatThreads, 0, stream>>>(a);
  else
    pack_kernel<kAgThreads, 1, 1><<<grid, kAgThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

constexpr size_t kBulkSmem = (size_t)TIDE_BULK_STAGES * TIDE_BULK_CHUNK + 8 * (TIDE_BULK_STAGES + 1);

cudaError_t launch_ag_bulk(const AgArgs& a, int grid, bool to_buf, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  auto k = to_buf ? ag_bulk_kernel<true> : ag_bulk_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
  if (e != cudaSuccess) return e;
  k<<<grid, 32, kBulkSmem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rs_bulk(const RsArgs& a, int grid, cudaStream_t stream) {
  if (grid <= 0 || a.num_tiles == 0) return cudaSuccess;
  const int N = a.num_ranks;
  const RsBulkGeom g = rs_bulk_geom(N, a.stage_bytes, a.rank_group);
  if (g.E < 8 || g.S < 2) return cudaErrorInvalidValue;
  if (g.groups > 1 && g.E > 8 * kRsBulkConsumers * kRsBulkGroupVecs) return cudaErrorInvalidValue;
  const size_t smem = (size_t)g.S * g.stage + 16 * (size_t)g.S + 8 * (size_t)N;
  cudaError_t e = cudaFuncSetAttribute(rs_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rs_bulk_kernel<<<grid, kRsBulkThreads, smem, stream>>>(a);
  return cudaGetLastError();
}


}  // namespace tide
