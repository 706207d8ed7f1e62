// Internal interface between the host layout descriptor / C ABI
// (layout.cpp, tide_api.cpp) and the CUDA kernels (kernels.cu).
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include <mutex>
#include <string>
#include <vector>

#include "tide.h"

namespace tide {

// One unit of kernel work: a contiguous run of `len` elements of one
// (parameter, rank) segment.  32 bytes, read once per tile by every CTA.
struct Tile {
  int64_t src;     // RS: element offset into grads[k][p] (same for every k)
                   // AG: element offset into the gathered buffer
  int64_t dst;     // RS: element offset into shards[r][p]; AG: into params[p]
  int32_t len;     // elements
  int32_t p;       // parameter
  int32_t r;       // rank whose shard / chunk the run belongs to
  uint32_t flags;  // kTileZero | kTileVec
};
static_assert(sizeof(Tile) == 32, "Tile is 32 bytes");

constexpr uint32_t kTileZero = 1u;  // RS only: write +0.0f (padding rows)
constexpr uint32_t kTileVec = 2u;   // source and destination allow 16-byte vectors

// Debug builds (-DTIDE_DEBUG=1) check every tile a kernel fetches against the
// extents of the buffers of its call before touching memory.
#ifndef TIDE_DEBUG
#define TIDE_DEBUG 0
#endif

// Element extents a tile may address: gradient / parameter storage of p
// (d0_p * inner_p), the fp32 shard of p (c_p * inner_p), and one rank-major
// buffer or slot (N * S).
struct Extents {
  const int64_t* grad_numel = nullptr;   // [P]
  const int64_t* shard_numel = nullptr;  // [P]
  int64_t buf_numel = 0;
  int32_t num_params = 0;
  int32_t num_ranks = 0;
};

// What a tile list feeds: its source and destination extents and the element
// alignment a 16-byte vector tile needs on each side.
enum TileKind : int { kKindRs = 0, kKindStagedRs = 1, kKindCopy = 2, kKindPack = 3 };

// True when `t` only addresses elements inside the extents of its kind:
// parameter and rank in range, non-negative offsets and length,
// src + len and dst + len within their buffers (the source of a zero tile
// is not read), known flags, zero tiles only in reduce-scatter lists, and the
// element alignment a vector tile's 16-byte accesses need.  Used by the
// kernels of a debug build and by tide_layout_check_tiles on the host.
__host__ __device__ inline bool tile_in_range(const Tile& t, int kind, const Extents& e) {
  if (t.p < 0 || t.p >= e.num_params || t.r < 0 || t.r >= e.num_ranks) return false;
  if (t.len < 0 || t.src < 0 || t.dst < 0) return false;
  if (t.flags & ~(kTileZero | kTileVec)) return false;
  const int64_t gn = e.grad_numel[t.p], sn = e.shard_numel[t.p], bn = e.buf_numel;
  int64_t src_n = 0, dst_n = 0, src_al = 8, dst_al = 8;
  switch (kind) {
    case kKindRs: src_n = gn; dst_n = sn; dst_al = 4; break;
    case kKindStagedRs: src_n = bn; dst_n = sn; dst_al = 4; break;
    case kKindCopy: src_n = bn; dst_n = gn; break;  // placement; staging runs it backwards
    case kKindPack: src_n = sn; dst_n = bn; src_al = 4; break;
    default: return false;
  }
  const bool zero = (t.flags & kTileZero) != 0;
  if (zero && kind != kKindRs && kind != kKindStagedRs) return false;
  if (!zero && t.src > src_n - t.len) return false;
  if (t.dst > dst_n - t.len) return false;
  if (t.flags & kTileVec) {
    if (!zero && t.src % src_al != 0) return false;
    if (t.dst % dst_al != 0) return false;
  }
  return true;
}

// Launch and tiling constants.  Each can be overridden at build time with the
// macro of the same name (used to sweep launch shapes).
#ifndef TIDE_RS_THREADS
#define TIDE_RS_THREADS 512
#endif
#ifndef TIDE_AG_THREADS
#define TIDE_AG_THREADS 512
#endif
#ifndef TIDE_AG_UNROLL
#define TIDE_AG_UNROLL 4
#endif
#ifndef TIDE_RS_TILE_READ_BYTES  // bf16 bytes read per RS tile across all N ranks
#define TIDE_RS_TILE_READ_BYTES 262144
#endif
#ifndef TIDE_AG_TILE_ELEMS
#define TIDE_AG_TILE_ELEMS 16384
#endif
#ifndef TIDE_AG_FAT_UNROLL  // 16-byte vectors a capped-mode placement thread loads before storing
#define TIDE_AG_FAT_UNROLL 8
#endif
#ifndef TIDE_PACK_FAT_UNROLL  // 8-element vectors a capped-mode pack thread loads before storing
#define TIDE_PACK_FAT_UNROLL 4
#endif
#ifndef TIDE_FAT_THREADS  // block of the CTA-capped mode: one fat CTA per occupied SM
#define TIDE_FAT_THREADS 1024
#endif
#ifndef TIDE_WARP_TILES  // 1: small capped grids hand tiles to single warps, not to whole CTAs
#define TIDE_WARP_TILES 1
#endif
#ifndef TIDE_RS_MIN_BLOCKS  // __launch_bounds__ min blocks per SM of the RS kernel
#define TIDE_RS_MIN_BLOCKS 1
#endif
constexpr int kRsThreads = TIDE_RS_THREADS;
constexpr int kAgThreads = TIDE_AG_THREADS;
constexpr int kFatThreads = TIDE_FAT_THREADS;
// Largest N the per-warp-tile capped reduce-scatter takes: its shared memory
// holds N source pointers per warp (16 KiB at 1024 threads).
constexpr int kRsWarpMaxRanks = 64;

// Arguments of the reduce-scatter kernel.  gtab is param-major
// (gtab[p * N + k] = rank k's gradient of p) so one tile's N pointers are
// contiguous; stab is rank-major (stab[r * P + p]).
struct RsArgs {
  const Tile* tiles;
  int64_t num_tiles;
  const uint16_t* const* gtab;
  float* const* stab;
  int32_t num_ranks;
  int32_t num_params;
  float scale;
  // bulk-staged kernel only (see AgArgs); stage_bytes: target bytes of one
  // ring stage; rank_group: ranks per stage (0 or >= N: all N rank slices of
  // a chunk in one stage; G < N: a chunk spans ceil(N / G) stages)
  int32_t stage_bytes = 0;
  int32_t rank_group = 0;
  int* err = nullptr;
  uint64_t timeout_ns = 0;
  uint64_t test_stall_ns = 0;
  Extents ext;  // checked per tile in debug builds (unchecked when ext.grad_numel is null)
  int kind = kKindRs;
};

// All-gather input pack: stab[r * P + p] is rank r's fp32 shard of p (only
// the ranks being packed are read); buf is the rank-major bf16 buffer.
struct PackArgs {
  const Tile* tiles;
  int64_t num_tiles;
  const float* const* stab;
  uint16_t* buf;
  int32_t num_params;
  int* err = nullptr;
  Extents ext;
};

struct AgArgs {
  const Tile* tiles;
  int64_t num_tiles;
  const uint16_t* buf;
  uint16_t* const* ptab;
  // placement only: when set, rank r's block is read from bufs[r] (each a
  // whole N*S rank-major buffer, e.g. rank r's own buffer mapped from its
  // process) instead of from buf
  const uint16_t* const* bufs = nullptr;
  // bulk-copy kernel only: error word set when a bounded wait runs out,
  // the bound, and a test hook that makes the first wait run out
  int* err;
  uint64_t timeout_ns;
  uint64_t test_stall_ns;
  Extents ext;
};

#ifndef TIDE_BULK_STAGES
#define TIDE_BULK_STAGES 4
#endif
#ifndef TIDE_BULK_CHUNK  // bytes per bulk copy (multiple of 16)
#define TIDE_BULK_CHUNK 16384
#endif
// TMA-staged reduce-scatter: bytes of one rank's slice of a chunk (over
// every SM / capped), and the stage size of rank-group staging.
#ifndef TIDE_RS_BULK_SLICE
#define TIDE_RS_BULK_SLICE 4096
#endif
#ifndef TIDE_RS_BULK_SLICE_CAPPED
#define TIDE_RS_BULK_SLICE_CAPPED 8192
#endif
#ifndef TIDE_RS_BULK_GROUP_STAGE
#define TIDE_RS_BULK_GROUP_STAGE 65536
#endif
#ifndef TIDE_RS_BULK_MIN_STAGE  // smallest stage when a chunk's N slices fit one (over every SM)
#define TIDE_RS_BULK_MIN_STAGE 65536
#endif
#ifndef TIDE_BULK_TIMEOUT_NS  // bound of every mbarrier wait of the bulk kernel
#define TIDE_BULK_TIMEOUT_NS 2000000000ull
#endif
// Error bits OR-ed into the device error word.
constexpr int kDevErrTimeout = 1;  // a bounded wait ran out
constexpr int kDevErrRange = 2;    // debug builds: a tile failed tile_in_range and was skipped

// A capped grid of at most half the device's SMs.  Each SM's own throughput
// bounds such a grid, so its fat CTAs hand tiles to single warps, which run
// out of step (one warp adds while the others' loads are in flight); larger
// grids are bound by HBM, where whole-CTA tiles stream better.
inline bool small_fat_grid(bool fat, int grid, int sms) { return TIDE_WARP_TILES && fat && 2 * (int64_t)grid <= sms; }

// Kernel launchers (kernels.cu).  Return the launch's cudaError_t.  `fat`
// selects the kFatThreads-wide CTA used by the CTA-capped mode: a capped CTA
// takes its SM away from full-SM compute kernels anyway, so it brings as many
// loads in flight as one SM holds.  `sms`: the device's SM count; a small
// capped grid (small_fat_grid) hands its tiles to single warps.
cudaError_t launch_rs(const RsArgs& a, int grid, bool fat, int sms, cudaStream_t stream);
cudaError_t launch_ag(const AgArgs& a, int grid, bool fat, int sms, cudaStream_t stream);
// The placement kernel run backwards (parameter storage -> rank-major
// buffer): Slot-Reuse staging of gradients.  `buf` is written.
cudaError_t launch_stage(const AgArgs& a, int grid, bool fat, int sms, cudaStream_t stream);
// Bulk-copy (TMA engine) placement / staging: one issuing lane per CTA,
// shared-memory ring of TIDE_BULK_STAGES x TIDE_BULK_CHUNK bytes.
cudaError_t launch_ag_bulk(const AgArgs& a, int grid, bool to_buf, cudaStream_t stream);
// Bulk-staged reduce-scatter (TMA engine): one CTA per SM, rank slices staged
// in shared memory by a producer warp; N <= kRsBulkMaxRanks.
constexpr int kRsBulkMaxRanks = 1024;  // bulk RS runs for N <= kRsBulkMaxRanks / 2
constexpr int kRsBulkThreads = 288;
cudaError_t launch_rs_bulk(const RsArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_pack(const PackArgs& a, int grid, bool fat, int sms, cudaStream_t stream);
int rs_block(bool fat);
int ag_block(bool fat);
int pk_block(bool fat);
// Resident CTAs per SM of each kernel for `num_ranks` (RS) at its block size.
size_t rs_smem_bytes(int32_t num_ranks);

// Device-side pointer table, cached by content.
struct PtrSlot {
  // identity of the cached table: tag (operation), rank, hash and the
  // caller's raw pointer arrays back to back
  uintptr_t tag = 0;
  intptr_t rank = 0;
  uint64_t hash = 0;
  size_t na = 0, nb = 0;
  std::vector<uintptr_t> key;
  void** d_table = nullptr;     // device copy
  void** h_staging = nullptr;   // pinned staging for the upload
  size_t capacity = 0;          // entries
  cudaEvent_t upload_ev = nullptr;
  cudaEvent_t use_ev = nullptr;
  cudaStream_t upload_stream = nullptr;
  cudaStream_t use_stream = nullptr;  // stream of the last kernel that read the table
  bool use_recorded = false;          // use_ev / use_stream are set (stream 0 is a valid stream)
  bool graph_pinned = false;          // read by a captured CUDA graph: never rewritten
  bool used = false;
  uint64_t last_use = 0;
};
constexpr int kPtrSlots = 8;

}  // namespace tide

struct tide_layout_s {
  uint64_t serial = 0;  // unique per layout within the process, never reused
  int32_t num_ranks = 0;
  int32_t num_params = 0;
  int64_t align = 8;
  std::vector<int64_t> d0, inner, chunk, shard_numel, offset;
  int64_t block_numel = 0;  // S
  // RS and pack tiles are rank-major: rank r's tiles are
  // [rank_begin[r], rank_begin[r + 1]) of their list.
  std::vector<tide::Tile> rs_tiles, ag_tiles, pk_tiles, st_tiles;
  std::vector<int64_t> rs_rank_begin, pk_rank_begin;
  tide_mode_t mode = TIDE_MODE_UNCAPPED;
  int32_t cta_cap = 0;

  // device state, created on first compute call
  int device = -1;
  tide::Tile* d_rs_tiles = nullptr;
  tide::Tile* d_ag_tiles = nullptr;
  tide::Tile* d_pk_tiles = nullptr;
  tide::Tile* d_st_tiles = nullptr;  // RS tiles whose sources are slot offsets
  int num_sms = 0;
  int* d_err = nullptr;         // device error word (bounded waits; range checks of debug builds)
  int64_t* d_extents = nullptr;  // [2P]: d0_p*inner_p, then c_p*inner_p
  // The tile lists and error word are uploaded on the stream of the first
  // compute call, from pinned staging kept until destroy; calls on other
  // streams wait on tables_ev until it has been seen complete.
  void* h_tile_staging = nullptr;
  cudaEvent_t tables_ev = nullptr;
  cudaStream_t tables_stream = nullptr;
  bool tables_resident = false;
  int64_t test_stall_ns = 0;    // test hook of the bounded waits
  int max_pitch = 0;
  tide::PtrSlot slots[tide::kPtrSlots];
  uint64_t use_counter = 0;
  std::mutex mu;
};

namespace tide {
tide_status_t set_error(tide_status_t st, const std::string& msg);
tide_status_t cuda_fail(cudaError_t e, const char* what);
int grid_for(int64_t tiles, tide_mode_t mode, int32_t cap, int sms, int per_sm);
int grid_of(const tide_layout_s* l, int64_t tiles, int per_sm);
}  // namespace tide
