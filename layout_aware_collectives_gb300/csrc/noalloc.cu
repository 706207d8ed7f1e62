// Reduce-scatter entry point that allocates no memory.
//
// The regular tide_rs_bf16_to_fp32 keeps its tile list and pointer tables in
// device memory it allocates (cudaMalloc, plus pinned staging from
// cudaMallocHost) on a layout's first call.  Some callers cannot allow that:
// a framework whose caching allocator owns all device memory and must not
// see allocations it does not track, a process running under a hard
// device-memory cap with every byte already reserved, or a step that cannot
// absorb the device-wide synchronisation a later cudaFree implies.  Layouts
// are built on the host without any CUDA call, so with this entry point such
// a caller runs the whole reduce-scatter without a single allocation.
//
// The kernel's scratch (tile list + gradient and shard pointer tables) lives
// in one file-scope __device__ array of kNoallocScratchBytes that every GPU
// loading this library holds until the process exits.
#include <cuda.h>  // driver-API types only; the entry points are fetched through the runtime
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "tide_internal.h"

namespace tide {
namespace {

constexpr size_t kNoallocScratchBytes = TIDE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// What one device's array holds: the tile list of layout `serial` and a
// pointer table, both copied on `stream`.  A later call on the same stream
// with the same layout and pointers skips the copies, since stream order
// already puts them before its kernel (a stream handle is only handed out
// again after the destroyed stream's work has completed).
struct Held {
  uint64_t serial = 0;  // 0: nothing known to be there
  cudaStream_t stream = nullptr;
  std::vector<const void*> table;
};

// Per device: the array's device address in the current CUDA context (in
// host code the symbol name is only a host-side stand-in, never a device
// address) and what the array holds.  Both belong to one context: after a
// cudaDeviceReset the module is loaded again, so the address may differ and
// the contents are gone; a new context id clears them.  `mu` is held from
// the check through the kernel launch, so copying calls serialise per device
// and never across devices.
struct DeviceState {
  std::mutex mu;
  void* addr = nullptr;
  unsigned long long ctx = 0;  // id of the context `addr` and `held` belong to
  int sms = 0;                 // the device's SM count
  Held held;
};
DeviceState g_dev[kMaxDevices];

// Id of the calling thread's current context (unique for the process's
// lifetime), 0 if none is current or the driver cannot tell.
using CtxGetCurrent = CUresult (*)(CUcontext*);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_entry_once;
CtxGetCurrent g_ctx_get_current = nullptr;
CtxGetId g_ctx_get_id = nullptr;

unsigned long long current_context_id() {
  std::call_once(g_entry_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = (CtxGetCurrent)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = (CtxGetId)f;
    cudaGetLastError();
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
  if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The current device's state, with its `mu` locked by `lock` and its address
// valid for the current context.
tide_status_t device_state(std::unique_lock<std::mutex>* lock, DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(TIDE_ERR_UNSUPPORTED, "device ordinal beyond the no-allocation table");
  DeviceState& d = g_dev[dev];
  *lock = std::unique_lock<std::mutex>(d.mu);
  unsigned long long ctx = current_context_id();
  if (!d.addr || ctx == 0 || ctx != d.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the runtime's context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    ctx = current_context_id();
    if (ctx == 0 || ctx != d.ctx) d.held = Held();  // another context: the contents are not ours
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
    d.addr = p;
    d.ctx = ctx;
  }
  *out = &d;
  return TIDE_OK;
}

tide_status_t check(const void* p, int64_t numel, const char* what, int64_t i) {
  if (numel == 0) return TIDE_OK;
  if (!p) return set_error(TIDE_ERR_INVALID_ARG, std::string(what) + "[" + std::to_string(i) + "] is NULL");
  if ((uintptr_t)p & 15u)
    return set_error(TIDE_ERR_MISALIGNED,
                     std::string(what) + "[" + std::to_string(i) + "] is not 16-byte aligned");
  return TIDE_OK;
}

}  // namespace
}  // namespace tide

using namespace tide;

extern "C" TIDE_API tide_status_t tide_rs_bf16_to_fp32_noalloc(tide_layout_t l,
                                                               const uint16_t* const* grads,
                                                               float* const* shards, float scale,
                                                               cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t N = l->num_ranks, P = l->num_params;
  if (P > 0 && (!grads || !shards)) return set_error(TIDE_ERR_INVALID_ARG, "pointer table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "reduce-scatter has no copy-engine mode");
  for (int64_t i = 0; i < (int64_t)N * P; ++i) {
    tide_status_t st = check(grads[i], l->d0[i % P] * l->inner[i % P], "grads", i);
    if (st == TIDE_OK) st = check(shards[i], l->shard_numel[i % P], "shards", i);
    if (st != TIDE_OK) return st;
  }
  if (l->rs_tiles.empty()) return TIDE_OK;

  const size_t tile_bytes = sizeof(Tile) * l->rs_tiles.size();
  const size_t table_bytes = sizeof(void*) * 2 * (size_t)N * P;
  if (tile_bytes + table_bytes > kNoallocScratchBytes)
    return set_error(TIDE_ERR_INVALID_ARG,
                     "layout needs " + std::to_string(tile_bytes + table_bytes) +
                         " bytes of scratch (tile list + pointer tables); the no-allocation "
                         "entry point holds at most " + std::to_string(kNoallocScratchBytes));
  // Pageable copies cannot live in a CUDA graph (the host table is gone at
  // replay), so a capture is refused before anything is enqueued.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return set_error(TIDE_ERR_UNSUPPORTED,
                     "the no-allocation entry point copies its tables from pageable host memory "
                     "and cannot be captured into a CUDA graph");
  std::unique_lock<std::mutex> dev_lock;
  DeviceState* ds = nullptr;
  tide_status_t st = device_state(&dev_lock, &ds);
  if (st != TIDE_OK) return st;

  const int64_t tiles = (int64_t)l->rs_tiles.size();
  // the load/store kernel in every mode: `cap` CTAs when capped, else one per tile
  const tide_mode_t mode = l->mode == TIDE_MODE_CAPPED ? TIDE_MODE_CAPPED : TIDE_MODE_UNCAPPED;
  const int grid = grid_for(tiles, mode, l->cta_cap, 0, 0);

  // Scratch layout: [tile list][param-major gradient table][rank-major shard table].
  std::vector<const void*> table(2 * (size_t)N * P);
  for (int32_t p = 0; p < P; ++p)
    for (int32_t k = 0; k < N; ++k) table[(size_t)p * N + k] = grads[(size_t)k * P + p];
  for (int64_t i = 0; i < (int64_t)N * P; ++i) table[(size_t)N * P + i] = shards[i];
  unsigned char* base = (unsigned char*)ds->addr;
  Held& held = ds->held;
  const bool same_tiles = held.serial == l->serial && held.stream == stream;
  const bool same_table = same_tiles && held.table == table;
  // Pageable sources: each copy returns once the driver holds its own copy of
  // the bytes, so the host vectors may go out of scope after the calls.  (The
  // copy waits for the stream's earlier work, so a call that copies blocks
  // the host until then; a repeated call copies nothing and returns at once.)
  cudaError_t e = cudaSuccess;
  if (!same_tiles) {
    held.serial = 0;
    e = cudaMemcpyAsync(base, l->rs_tiles.data(), tile_bytes, cudaMemcpyHostToDevice, stream);
  }
  if (e == cudaSuccess && !same_table) {
    held.serial = 0;
    e = cudaMemcpyAsync(base + tile_bytes, table.data(), table_bytes, cudaMemcpyHostToDevice, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "copy of the tables into the no-allocation scratch");
  if (!same_table) {
    held.serial = l->serial;
    held.stream = stream;
    held.table.swap(table);
  }

  RsArgs a;
  a.tiles = (const Tile*)base;
  a.num_tiles = tiles;
  a.gtab = (const uint16_t* const*)(base + tile_bytes);
  a.stab = (float* const*)(base + tile_bytes) + (size_t)N * P;
  a.num_ranks = N;
  a.num_params = P;
  a.scale = scale;
  e = launch_rs(a, grid, l->mode == TIDE_MODE_CAPPED, ds->sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter kernel launch");
  return TIDE_OK;
}
