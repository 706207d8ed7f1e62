// C ABI compute entry points: argument validation, lazy device set-up of a
// layout, the device pointer-table cache, mode dispatch (uncapped / CTA-capped
// kernels, copy-engine placement) and the launches.
#include <algorithm>
#include <cstring>

#include "tide_internal.h"

namespace tide {
namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

#define TIDE_CUDA(call, what)                 \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

struct DeviceShape {
  int sms = 0;
};

tide_status_t query_device(DeviceShape* d) {
  int dev = 0;
  TIDE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  TIDE_CUDA(cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev),
            "cudaDeviceGetAttribute(MultiProcessorCount)");
  return TIDE_OK;
}

}  // namespace

// Grid of one launch over `tiles` tiles.  Capped modes launch `cap` CTAs
// that loop over the list.  Otherwise the TMA-staged reduce-scatter
// (per_sm > 0: its ring fills an SM) launches per_sm CTAs per SM, and every
// other kernel one CTA per tile, so the hardware block scheduler hands tiles
// out in list order as CTAs retire; on GB300 that streams 3-17% faster than
// SM-filling CTAs looping over the list (the loop stays: a grid below
// `tiles` is still correct).
int grid_for(int64_t tiles, tide_mode_t mode, int32_t cap, int sms, int per_sm) {
  if (tiles <= 0) return 0;
  const bool capped = mode == TIDE_MODE_CAPPED || (mode == TIDE_MODE_BULK && cap > 0);
  const int64_t g = capped ? (int64_t)cap : per_sm > 0 ? (int64_t)sms * per_sm : tiles;
  return (int)std::min<int64_t>(std::min<int64_t>(tiles, g), INT32_MAX);
}

namespace {

bool rs_uses_bulk(const tide_layout_s* l) {
  // N <= 512 keeps rank slices of at least 96 elements in a 96 KiB stage and
  // the N source pointers within the CTA's shared memory
  return l->mode == TIDE_MODE_BULK && l->num_ranks <= kRsBulkMaxRanks / 2;
}

// True while `stream` is being captured into a CUDA graph.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return st == cudaStreamCaptureStatusActive;
}

void release_device(tide_layout_s* l) {
  for (PtrSlot& s : l->slots) {
    if (s.use_ev && s.use_recorded) cudaEventSynchronize(s.use_ev);
    if (s.d_table) cudaFree(s.d_table);
    if (s.h_staging) cudaFreeHost(s.h_staging);
    if (s.upload_ev) cudaEventDestroy(s.upload_ev);
    if (s.use_ev) cudaEventDestroy(s.use_ev);
    s = PtrSlot();
  }
  Tile** lists[4] = {&l->d_rs_tiles, &l->d_ag_tiles, &l->d_pk_tiles, &l->d_st_tiles};
  for (Tile** t : lists) {
    if (*t) cudaFree(*t);
    *t = nullptr;
  }
  if (l->d_err) cudaFree(l->d_err);
  l->d_err = nullptr;
  if (l->d_extents) cudaFree(l->d_extents);
  l->d_extents = nullptr;
  if (l->tables_ev) {
    cudaEventSynchronize(l->tables_ev);  // the upload reads the staging
    cudaEventDestroy(l->tables_ev);
  }
  l->tables_ev = nullptr;
  if (l->h_tile_staging) cudaFreeHost(l->h_tile_staging);
  l->h_tile_staging = nullptr;
  l->tables_stream = nullptr;
  l->tables_resident = false;
  cudaGetLastError();  // leave no error of the clean-up behind
}

tide_status_t bind_device(tide_layout_s* l, int dev, cudaStream_t stream);

// Bind the layout to the current device on first use (query the SM count,
// upload the tile lists on `stream`); later, order a call on another stream
// after that upload until it has been seen complete.  On failure everything
// allocated so far is released and the layout stays unbound.
tide_status_t ensure_device(tide_layout_s* l, cudaStream_t stream) {
  int dev = 0;
  TIDE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (l->device >= 0) {
    if (dev != l->device)
      return set_error(TIDE_ERR_INVALID_ARG, "layout is bound to device " + std::to_string(l->device) +
                                                 " but device " + std::to_string(dev) + " is current");
    if (!l->tables_resident && stream != l->tables_stream && !capturing(stream)) {
      const cudaError_t q = cudaEventQuery(l->tables_ev);
      if (q == cudaSuccess) {
        l->tables_resident = true;
      } else if (q == cudaErrorNotReady) {
        TIDE_CUDA(cudaStreamWaitEvent(stream, l->tables_ev, 0), "cudaStreamWaitEvent");
      } else {
        return cuda_fail(q, "cudaEventQuery(tile-list upload)");
      }
    }
    return TIDE_OK;
  }
  if (capturing(stream))
    return set_error(TIDE_ERR_UNSUPPORTED,
                     "the layout's first compute call sets it up on the device and cannot be captured; "
                     "make one call on this stream before capturing");
  tide_status_t st = bind_device(l, dev, stream);
  if (st != TIDE_OK) release_device(l);
  return st;
}

tide_status_t bind_device(tide_layout_s* l, int dev, cudaStream_t stream) {
  DeviceShape d;
  tide_status_t st = query_device(&d);
  if (st != TIDE_OK) return st;
  TIDE_CUDA(cudaDeviceGetAttribute(&l->max_pitch, cudaDevAttrMaxPitch, dev),
            "cudaDeviceGetAttribute(MaxPitch)");
  struct {
    const std::vector<Tile>* host;
    Tile** dev;
    const char* what;
  } lists[4] = {{&l->rs_tiles, &l->d_rs_tiles, "reduce-scatter tile list"},
                {&l->ag_tiles, &l->d_ag_tiles, "placement tile list"},
                {&l->pk_tiles, &l->d_pk_tiles, "pack tile list"},
                {&l->st_tiles, &l->d_st_tiles, "staged reduce-scatter tile list"}};
  // One pinned staging buffer for the four lists and the extents: the copies
  // are then asynchronous (a pageable source would make the host wait for
  // the stream).
  const size_t P = (size_t)l->num_params;
  size_t total = 0;
  for (auto& t : lists) total += t.host->size();
  TIDE_CUDA(cudaMallocHost(&l->h_tile_staging, sizeof(Tile) * total + 2 * sizeof(int64_t) * std::max<size_t>(1, P)),
            "cudaMallocHost(tile-list staging)");
  Tile* staged = (Tile*)l->h_tile_staging;
  for (auto& t : lists) {
    TIDE_CUDA(cudaMalloc((void**)t.dev, sizeof(Tile) * std::max<size_t>(1, t.host->size())),
              "cudaMalloc(tile list)");
    if (!t.host->empty()) {
      std::memcpy(staged, t.host->data(), sizeof(Tile) * t.host->size());
      TIDE_CUDA(cudaMemcpyAsync(*t.dev, staged, sizeof(Tile) * t.host->size(), cudaMemcpyHostToDevice, stream),
                t.what);
      staged += t.host->size();
    }
  }
  // extents the debug build's kernels check every tile against
  int64_t* ext = (int64_t*)staged;
  for (size_t p = 0; p < P; ++p) {
    ext[p] = l->d0[p] * l->inner[p];
    ext[P + p] = l->shard_numel[p];
  }
  TIDE_CUDA(cudaMalloc((void**)&l->d_extents, 2 * sizeof(int64_t) * std::max<size_t>(1, P)),
            "cudaMalloc(extents)");
  if (P)
    TIDE_CUDA(cudaMemcpyAsync(l->d_extents, ext, 2 * sizeof(int64_t) * P, cudaMemcpyHostToDevice, stream),
              "extents");
  TIDE_CUDA(cudaMalloc((void**)&l->d_err, sizeof(int)), "cudaMalloc(error word)");
  TIDE_CUDA(cudaMemsetAsync(l->d_err, 0, sizeof(int), stream), "cudaMemsetAsync(error word)");
  TIDE_CUDA(cudaEventCreateWithFlags(&l->tables_ev, cudaEventDisableTiming), "cudaEventCreate");
  TIDE_CUDA(cudaEventRecord(l->tables_ev, stream), "cudaEventRecord");
  l->tables_stream = stream;
  for (PtrSlot& s : l->slots) {
    TIDE_CUDA(cudaEventCreateWithFlags(&s.upload_ev, cudaEventDisableTiming), "cudaEventCreate");
    TIDE_CUDA(cudaEventCreateWithFlags(&s.use_ev, cudaEventDisableTiming), "cudaEventCreate");
  }
  l->num_sms = d.sms;
  l->device = dev;
  return TIDE_OK;
}

// Identity of a pointer-table request: the caller's raw pointer arrays (one
// or two), with the operation tag and rank.  The hash is FNV-1a over the
// pointer values; a hit is confirmed by comparing the arrays themselves.
struct TableKey {
  uintptr_t tag;
  intptr_t rank;
  const void* const* a;
  size_t na;
  const void* const* b;
  size_t nb;
  uint64_t hash;
};

TableKey make_key(uintptr_t tag, intptr_t rank, const void* const* a, size_t na, const void* const* b,
                  size_t nb) {
  uint64_t h = 1469598103934665603ull ^ (tag * 0x9E3779B97F4A7C15ull) ^ (uint64_t)rank;
  for (size_t i = 0; i < na; ++i) h = (h ^ (uint64_t)(uintptr_t)a[i]) * 1099511628211ull;
  for (size_t i = 0; i < nb; ++i) h = (h ^ (uint64_t)(uintptr_t)b[i]) * 1099511628211ull;
  return TableKey{tag, rank, a, na, b, nb, h};
}

bool same_key(const PtrSlot& s, const TableKey& k) {
  return s.used && s.hash == k.hash && s.tag == k.tag && s.rank == k.rank && s.na == k.na &&
         s.nb == k.nb && (k.na == 0 || !std::memcmp(s.key.data(), k.a, k.na * sizeof(void*))) &&
         (k.nb == 0 || !std::memcmp(s.key.data() + k.na, k.b, k.nb * sizeof(void*)));
}

// True when a slot already holds this exact pointer set: the pointers were
// validated when the slot was filled, so a hit skips validation.
bool cached(const tide_layout_s* l, const TableKey& key) {
  for (const PtrSlot& s : l->slots)
    if (same_key(s, key)) return true;
  return false;
}

// Device copy of a pointer table, cached by content: steady-state training
// passes the same buffers every step, so a hit costs a hash and array
// comparison and, when the stream changed, a stream-ordering wait.  On a miss
// `build(dst)` writes the n_entries table entries in device order.
template <typename Build>
tide_status_t acquire_table(tide_layout_s* l, const TableKey& key, size_t n_entries, Build&& build,
                            cudaStream_t stream, PtrSlot** out) {
  PtrSlot* hit = nullptr;
  for (PtrSlot& s : l->slots)
    if (same_key(s, key)) {
      hit = &s;
      break;
    }
  const bool cap = capturing(stream);
  if (hit) {
    // Inside a capture the table was uploaded by an earlier call on this
    // stream (required), and no host-side event is recorded or waited on.
    if (!cap && hit->upload_stream != stream)
      TIDE_CUDA(cudaStreamWaitEvent(stream, hit->upload_ev, 0), "cudaStreamWaitEvent");
    // One event tracks the slot's last reader, so a reader on another stream
    // is ordered after the previous one: the event then covers both, and an
    // eviction that waits on it cannot overwrite a table still being read.
    if (!cap && hit->use_recorded && hit->use_stream != stream)
      TIDE_CUDA(cudaStreamWaitEvent(stream, hit->use_ev, 0), "cudaStreamWaitEvent");
    *out = hit;
    return TIDE_OK;
  }
  if (cap)
    return set_error(TIDE_ERR_UNSUPPORTED,
                     "pointer set used for the first time inside a stream capture; make one call "
                     "with these pointers on this stream before capturing");
  PtrSlot* s = nullptr;  // a free slot, else the least recently used one no graph reads
  for (PtrSlot& c : l->slots) {
    if (c.graph_pinned) continue;
    if (!c.used) {
      s = &c;
      break;
    }
    if (!s || c.last_use < s->last_use) s = &c;
  }
  if (!s)
    return set_error(TIDE_ERR_UNSUPPORTED,
                     "every pointer-table slot of this layout is read by a captured CUDA graph");
  // Kernels that read this slot's previous table, and its previous upload
  // from the staging buffer, must be done before either is overwritten.
  if (s->used && s->use_recorded) TIDE_CUDA(cudaEventSynchronize(s->use_ev), "cudaEventSynchronize");
  if (s->used && !s->use_recorded) TIDE_CUDA(cudaEventSynchronize(s->upload_ev), "cudaEventSynchronize");
  s->used = false;
  s->use_stream = nullptr;
  s->use_recorded = false;
  // A slot is allocated on its first use at the largest table any operation
  // needs (2*N*P entries), so no later call frees device memory (a cudaFree
  // would synchronise the device).
  const size_t n = std::max<size_t>(1, 2 * (size_t)l->num_ranks * (size_t)l->num_params);
  if (n_entries > n) return set_error(TIDE_ERR_INVALID_ARG, "pointer table larger than 2*N*P entries");
  if (s->capacity == 0) {
    TIDE_CUDA(cudaMalloc((void**)&s->d_table, n * sizeof(void*)), "cudaMalloc(pointer table)");
    TIDE_CUDA(cudaMallocHost((void**)&s->h_staging, n * sizeof(void*)),
              "cudaMallocHost(pointer table staging)");
    s->capacity = n;
  }
  if (n_entries) {
    build(s->h_staging);
    TIDE_CUDA(cudaMemcpyAsync(s->d_table, s->h_staging, n_entries * sizeof(void*), cudaMemcpyHostToDevice,
                              stream),
              "upload of the pointer table");
  }
  TIDE_CUDA(cudaEventRecord(s->upload_ev, stream), "cudaEventRecord");
  s->upload_stream = stream;
  s->tag = key.tag;
  s->rank = key.rank;
  s->hash = key.hash;
  s->na = key.na;
  s->nb = key.nb;
  s->key.resize(key.na + key.nb);
  if (key.na) std::memcpy(s->key.data(), key.a, key.na * sizeof(void*));
  if (key.nb) std::memcpy(s->key.data() + key.na, key.b, key.nb * sizeof(void*));
  s->used = true;
  *out = s;
  return TIDE_OK;
}

tide_status_t mark_used(tide_layout_s* l, PtrSlot* s, cudaStream_t stream) {
  s->last_use = ++l->use_counter;
  if (capturing(stream)) {  // a graph may replay this launch at any time from now on
    s->graph_pinned = true;
    return TIDE_OK;
  }
  TIDE_CUDA(cudaEventRecord(s->use_ev, stream), "cudaEventRecord");
  s->use_stream = stream;
  s->use_recorded = true;
  return TIDE_OK;
}

tide_status_t check_ptr(const void* p, int64_t numel, const char* what, int64_t i) {
  if (numel == 0) return TIDE_OK;
  if (!p) return set_error(TIDE_ERR_INVALID_ARG, std::string(what) + "[" + std::to_string(i) + "] is NULL");
  if (!aligned16(p))
    return set_error(TIDE_ERR_MISALIGNED,
                     std::string(what) + "[" + std::to_string(i) + "] is not 16-byte aligned");
  return TIDE_OK;
}

// Copy-engine placement: per parameter one strided 2-D copy for the ranks
// that own a full chunk (rank r's chunk is contiguous in both the buffer, at
// r*S + o_p, and the parameter, at r*c*inner) and one plain copy for the
// rank that owns a partial chunk.  to_buf runs the copies backwards
// (parameter storage -> rank-major buffer: Slot-Reuse staging).
tide_status_t copy_engine(tide_layout_s* l, uint16_t* buf, uint16_t* const* params, bool to_buf,
                          cudaStream_t stream) {
  const int64_t S = l->block_numel;
  for (int32_t p = 0; p < l->num_params; ++p) {
    const int64_t c = l->chunk[p], inner = l->inner[p], d0 = l->d0[p];
    if (c == 0 || inner == 0) continue;
    const int64_t full = std::min<int64_t>(l->num_ranks, d0 / c);
    const size_t width = (size_t)(c * inner) * 2;
    const size_t bpitch = (size_t)S * 2;
    uint16_t* b = buf + l->offset[p];
    uint16_t* q = params[p];
    if (full > 0) {
      if (bpitch <= (size_t)l->max_pitch && full > 1) {
        cudaError_t e = to_buf ? cudaMemcpy2DAsync(b, bpitch, q, width, width, (size_t)full,
                                                   cudaMemcpyDeviceToDevice, stream)
                               : cudaMemcpy2DAsync(q, width, b, bpitch, width, (size_t)full,
                                                   cudaMemcpyDeviceToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
      } else {
        for (int64_t r = 0; r < full; ++r) {
          uint16_t* x = b + r * S;
          uint16_t* y = q + r * c * inner;
          TIDE_CUDA(cudaMemcpyAsync(to_buf ? x : y, to_buf ? y : x, width, cudaMemcpyDeviceToDevice,
                                    stream),
                    "cudaMemcpyAsync");
        }
      }
    }
    const int64_t rows = d0 - full * c;
    if (rows > 0 && full < l->num_ranks) {
      uint16_t* x = b + full * S;
      uint16_t* y = q + full * c * inner;
      TIDE_CUDA(cudaMemcpyAsync(to_buf ? x : y, to_buf ? y : x, (size_t)(rows * inner) * 2,
                                cudaMemcpyDeviceToDevice, stream),
                "cudaMemcpyAsync");
    }
  }
  return TIDE_OK;
}

}  // namespace

Extents extents_of(const tide_layout_s* l) {
  Extents e;
  e.grad_numel = l->d_extents;
  e.shard_numel = l->d_extents + l->num_params;
  e.buf_numel = l->block_numel * l->num_ranks;
  e.num_params = l->num_params;
  e.num_ranks = l->num_ranks;
  return e;
}

int grid_of(const tide_layout_s* l, int64_t tiles, int per_sm) {
  return grid_for(tiles, l->mode, l->cta_cap, l->num_sms, per_sm);
}

}  // namespace tide

using namespace tide;

namespace tide {
namespace {

// Shared steps of the reduce-scatter entry points once arguments are
// validated: bind the device, fetch the cached device pointer table (built
// by `build` on a miss: N*P source pointers param-major, then N*P shard
// pointers rank-major), launch.
template <typename Build>
tide_status_t run_rs(tide_layout_s* l, bool staged, int64_t t0, int64_t t1, const TableKey& key, Build&& build,
                     float scale, cudaStream_t stream) {
  if (t1 <= t0) return TIDE_OK;
  tide_status_t st = ensure_device(l, stream);
  if (st != TIDE_OK) return st;
  const int64_t NP = (int64_t)l->num_ranks * l->num_params;
  PtrSlot* slot = nullptr;
  st = acquire_table(l, key, (size_t)(2 * NP), build, stream, &slot);
  if (st != TIDE_OK) return st;
  RsArgs a;
  a.tiles = (staged ? l->d_st_tiles : l->d_rs_tiles) + t0;
  a.num_tiles = t1 - t0;
  a.gtab = (const uint16_t* const*)slot->d_table;
  a.stab = (float* const*)(slot->d_table + NP);
  a.num_ranks = l->num_ranks;
  a.num_params = l->num_params;
  a.scale = scale;
  a.err = l->d_err;
  a.timeout_ns = TIDE_BULK_TIMEOUT_NS;
  a.test_stall_ns = (uint64_t)l->test_stall_ns;
  a.ext = extents_of(l);
  a.kind = staged ? kKindStagedRs : kKindRs;
  // TMA-staged kernel.  Measured on GB300: rank slices of 4 KiB over every
  // SM (8 KiB when capped) keep the bulk-copy engine busy and smaller ones
  // do not, and 64 KiB stages (a 3-deep ring) beat 32 KiB ones (by 1-2% at
  // N = 8, 12% with rank groups) and 96 KiB ones.  When all N slices of a
  // chunk fit a stage of TIDE_RS_BULK_GROUP_STAGE bytes, one stage holds
  // them (at least TIDE_RS_BULK_MIN_STAGE bytes, so slices grow as N
  // shrinks); above that N a stage holds the slices of
  // TIDE_RS_BULK_GROUP_STAGE / slice ranks and a chunk spans consecutive
  // stages, so slices and ring depth no longer shrink as N grows.
  const int64_t slice_target = l->cta_cap > 0 ? TIDE_RS_BULK_SLICE_CAPPED : TIDE_RS_BULK_SLICE;
  const int64_t group = std::max<int64_t>(1, TIDE_RS_BULK_GROUP_STAGE / slice_target);
  if (l->num_ranks > group) {
    a.rank_group = (int32_t)group;
    a.stage_bytes = (int32_t)(group * slice_target);
  } else {
    a.rank_group = 0;
    a.stage_bytes = (int32_t)std::min<int64_t>(
        98304, std::max<int64_t>(TIDE_RS_BULK_MIN_STAGE,
                                 (int64_t)l->num_ranks * slice_target));
  }
  cudaError_t e = rs_uses_bulk(l) ? launch_rs_bulk(a, grid_of(l, t1 - t0, 1), stream)
                                  : launch_rs(a, grid_of(l, t1 - t0, 0), l->mode == TIDE_MODE_CAPPED, l->num_sms,
                                              stream);
  if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter kernel launch");
  return mark_used(l, slot, stream);
}

// Validation of N*P gradient pointers (rank-major) and of `nout` shard
// pointers (all ranks, or one rank's P).
tide_status_t check_rs_ptrs(const tide_layout_s* l, const uint16_t* const* grads, float* const* shards,
                            int64_t nout) {
  const int32_t N = l->num_ranks, P = l->num_params;
  for (int32_t k = 0; k < N; ++k)
    for (int32_t p = 0; p < P; ++p) {
      const int64_t i = (int64_t)k * P + p;
      tide_status_t st = check_ptr(grads[i], l->d0[p] * l->inner[p], "grads", i);
      if (st != TIDE_OK) return st;
    }
  for (int64_t i = 0, p = 0; i < nout; ++i, p = (p + 1 == P ? 0 : p + 1)) {
    tide_status_t st = check_ptr(shards[i], l->shard_numel[p], "shards", i);
    if (st != TIDE_OK) return st;
  }
  return TIDE_OK;
}

// Device table of a reduce-scatter: gradients param-major, then the shard
// table rank-major with the entries of ranks not written left null.
void build_rs_table(const tide_layout_s* l, int32_t rank, const uint16_t* const* grads, float* const* shards,
                    void** dst) {
  const int32_t N = l->num_ranks, P = l->num_params;
  const size_t NP = (size_t)N * P;
  for (int32_t p = 0; p < P; ++p)
    for (int32_t k = 0; k < N; ++k) dst[(size_t)p * N + k] = (void*)grads[(size_t)k * P + p];
  if (rank < 0) {
    std::memcpy(dst + NP, shards, NP * sizeof(void*));
  } else {
    std::memset(dst + NP, 0, NP * sizeof(void*));
    std::memcpy(dst + NP + (size_t)rank * P, shards, (size_t)P * sizeof(void*));
  }
}

// Placement (to_buf = false) or staging (to_buf = true) over the AG tile
// list: the bulk-copy kernel in TIDE_MODE_BULK, else the load/store kernel.
cudaError_t launch_copy(tide_layout_s* l, AgArgs& a, bool to_buf, cudaStream_t stream) {
  a.err = l->d_err;
  a.timeout_ns = TIDE_BULK_TIMEOUT_NS;
  a.test_stall_ns = (uint64_t)l->test_stall_ns;
  a.ext = extents_of(l);
  const bool capped = l->mode == TIDE_MODE_CAPPED;
  if (l->mode == TIDE_MODE_BULK)
    return launch_ag_bulk(a, grid_of(l, a.num_tiles, 0), to_buf, stream);
  return to_buf ? launch_stage(a, grid_of(l, a.num_tiles, 0), capped, l->num_sms, stream)
                : launch_ag(a, grid_of(l, a.num_tiles, 0), capped, l->num_sms, stream);
}

}  // namespace
}  // namespace tide

extern "C" {

void tide_layout_destroy(tide_layout_t l) {
  if (!l) return;
  if (l->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != l->device) cudaSetDevice(l->device);
    release_device(l);
    if (cur >= 0 && cur != l->device) cudaSetDevice(cur);
  }
  delete l;
}

tide_status_t tide_layout_launch_shape(tide_layout_t l, tide_op_t op, int32_t* grid, int32_t* block) {
  if (!l || !grid || !block) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  if (op < TIDE_OP_RS || op > TIDE_OP_STAGED_RS) return set_error(TIDE_ERR_INVALID_ARG, "unknown op");
  std::lock_guard<std::mutex> g(l->mu);
  DeviceShape d;
  tide_status_t st = query_device(&d);
  if (st != TIDE_OK) return st;
  const bool capped = l->mode == TIDE_MODE_CAPPED;
  const bool rs_like = op == TIDE_OP_RS || op == TIDE_OP_STAGED_RS;
  const int64_t tiles = op == TIDE_OP_RS          ? (int64_t)l->rs_tiles.size()
                        : op == TIDE_OP_STAGED_RS ? (int64_t)l->st_tiles.size()
                        : op == TIDE_OP_PACK      ? (int64_t)l->pk_tiles.size()
                                                  : (int64_t)l->ag_tiles.size();
  const bool bulk = l->mode == TIDE_MODE_BULK && (op == TIDE_OP_AG || op == TIDE_OP_STAGE);
  const bool rs_bulk = rs_like && rs_uses_bulk(l);
  const int per_sm = rs_bulk ? 1 : 0;
  *grid = l->mode == TIDE_MODE_COPY_ENGINE ? 0 : grid_for(tiles, l->mode, l->cta_cap, d.sms, per_sm);
  *block = rs_bulk ? kRsBulkThreads : rs_like ? rs_block(capped) : op == TIDE_OP_PACK ? pk_block(capped)
                   : bulk ? 32 : ag_block(capped);
  return TIDE_OK;
}

tide_status_t tide_rs_bf16_to_fp32(tide_layout_t l, const uint16_t* const* grads, float* const* shards,
                                   float scale, cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  if (l->num_params > 0 && (!grads || !shards))
    return set_error(TIDE_ERR_INVALID_ARG, "pointer table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "reduce-scatter has no copy-engine mode");
  const int64_t NP = (int64_t)l->num_ranks * l->num_params;
  const TableKey key = make_key(TIDE_OP_RS, -1, (const void* const*)grads, (size_t)NP,
                                (const void* const*)shards, (size_t)NP);
  if (!cached(l, key)) {
    tide_status_t st = check_rs_ptrs(l, grads, shards, NP);
    if (st != TIDE_OK) return st;
  }
  return run_rs(l, false, 0, (int64_t)l->rs_tiles.size(), key,
                [&](void** dst) { build_rs_table(l, -1, grads, shards, dst); }, scale, stream);
}

tide_status_t tide_rs_bf16_to_fp32_rank(tide_layout_t l, int32_t rank, const uint16_t* const* grads,
                                        float* const* shards, float scale, cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  if (rank < 0 || rank >= l->num_ranks) return set_error(TIDE_ERR_INVALID_ARG, "rank out of range");
  if (l->num_params > 0 && (!grads || !shards))
    return set_error(TIDE_ERR_INVALID_ARG, "pointer table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "reduce-scatter has no copy-engine mode");
  const int64_t NP = (int64_t)l->num_ranks * l->num_params;
  const TableKey key = make_key(TIDE_OP_RS, rank, (const void* const*)grads, (size_t)NP,
                                (const void* const*)shards, (size_t)l->num_params);
  if (!cached(l, key)) {
    tide_status_t st = check_rs_ptrs(l, grads, shards, l->num_params);
    if (st != TIDE_OK) return st;
  }
  return run_rs(l, false, l->rs_rank_begin[rank], l->rs_rank_begin[rank + 1], key,
                [&](void** dst) { build_rs_table(l, rank, grads, shards, dst); }, scale, stream);
}

tide_status_t tide_ag_place(tide_layout_t l, const uint16_t* gathered, uint16_t* const* params,
                            cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t P = l->num_params;
  if (P > 0 && !params) return set_error(TIDE_ERR_INVALID_ARG, "params table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  tide_status_t st = check_ptr(gathered, l->block_numel * l->num_ranks, "gathered", 0);
  if (st != TIDE_OK) return st;
  for (int32_t p = 0; p < P; ++p) {
    st = check_ptr(params[p], l->d0[p] * l->inner[p], "params", p);
    if (st != TIDE_OK) return st;
  }
  if (l->ag_tiles.empty()) return TIDE_OK;
  st = ensure_device(l, stream);
  if (st != TIDE_OK) return st;
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return copy_engine(l, const_cast<uint16_t*>(gathered), params, false, stream);

  const TableKey key = make_key(TIDE_OP_AG, 0, (const void* const*)params, (size_t)P, nullptr, 0);
  PtrSlot* slot = nullptr;
  st = acquire_table(
      l, key, (size_t)P, [&](void** dst) { std::memcpy(dst, params, (size_t)P * sizeof(void*)); }, stream,
      &slot);
  if (st != TIDE_OK) return st;

  AgArgs a;
  a.tiles = l->d_ag_tiles;
  a.num_tiles = (int64_t)l->ag_tiles.size();
  a.buf = gathered;
  a.ptab = (uint16_t* const*)slot->d_table;
  cudaError_t e = launch_copy(l, a, false, stream);
  if (e != cudaSuccess) return cuda_fail(e, "placement kernel launch");
  return mark_used(l, slot, stream);
}

tide_status_t tide_ag_place_ranks(tide_layout_t l, const uint16_t* const* gathered, uint16_t* const* params,
                                  cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t N = l->num_ranks, P = l->num_params;
  if (!gathered) return set_error(TIDE_ERR_INVALID_ARG, "gathered table is NULL");
  if (P > 0 && !params) return set_error(TIDE_ERR_INVALID_ARG, "params table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  for (int32_t k = 0; k < N; ++k) {
    tide_status_t st = check_ptr(gathered[k], l->block_numel * N, "gathered", k);
    if (st != TIDE_OK) return st;
  }
  for (int32_t p = 0; p < P; ++p) {
    tide_status_t st = check_ptr(params[p], l->d0[p] * l->inner[p], "params", p);
    if (st != TIDE_OK) return st;
  }
  if (l->ag_tiles.empty()) return TIDE_OK;
  tide_status_t st = ensure_device(l, stream);
  if (st != TIDE_OK) return st;
  if (l->mode == TIDE_MODE_COPY_ENGINE) {  // one copy per (parameter, rank) with rows
    for (int32_t p = 0; p < P; ++p) {
      const int64_t c = l->chunk[p], inner = l->inner[p];
      for (int32_t r = 0; r < N; ++r) {
        const int64_t v = std::max<int64_t>(0, std::min<int64_t>(c, l->d0[p] - (int64_t)r * c)) * inner;
        if (v == 0) continue;
        TIDE_CUDA(cudaMemcpyAsync(params[p] + (int64_t)r * c * inner,
                                  gathered[r] + (int64_t)r * l->block_numel + l->offset[p], (size_t)v * 2,
                                  cudaMemcpyDeviceToDevice, stream),
                  "cudaMemcpyAsync");
      }
    }
    return TIDE_OK;
  }
  // device table: P parameter pointers, then the N rank buffers
  const TableKey key = make_key(TIDE_OP_AG, -2, (const void* const*)params, (size_t)P,
                                (const void* const*)gathered, (size_t)N);
  PtrSlot* slot = nullptr;
  st = acquire_table(
      l, key, (size_t)P + (size_t)N,
      [&](void** dst) {
        std::memcpy(dst, params, (size_t)P * sizeof(void*));
        std::memcpy(dst + P, gathered, (size_t)N * sizeof(void*));
      },
      stream, &slot);
  if (st != TIDE_OK) return st;
  AgArgs a;
  a.tiles = l->d_ag_tiles;
  a.num_tiles = (int64_t)l->ag_tiles.size();
  a.buf = gathered[0];
  a.ptab = (uint16_t* const*)slot->d_table;
  a.bufs = (const uint16_t* const*)(slot->d_table + P);
  a.err = l->d_err;
  a.timeout_ns = TIDE_BULK_TIMEOUT_NS;
  a.test_stall_ns = 0;
  a.ext = extents_of(l);
  // the load/store kernel in every mode (the TMA copies are for this
  // process's own memory): `cap` CTAs when capped, else one per tile
  const bool capped = l->mode == TIDE_MODE_CAPPED;
  const int grid = grid_for(a.num_tiles, capped ? TIDE_MODE_CAPPED : TIDE_MODE_UNCAPPED, l->cta_cap, l->num_sms, 0);
  cudaError_t e = launch_ag(a, grid, capped, l->num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "placement kernel launch");
  return mark_used(l, slot, stream);
}

tide_status_t tide_ag_pack_bf16(tide_layout_t l, int32_t rank, const float* const* shards,
                                uint16_t* gathered, cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t N = l->num_ranks, P = l->num_params;
  if (rank < -1 || rank >= N) return set_error(TIDE_ERR_INVALID_ARG, "rank out of range");
  if (P > 0 && !shards) return set_error(TIDE_ERR_INVALID_ARG, "shards table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "the pack casts on the SMs; no copy-engine mode");
  tide_status_t st = check_ptr(gathered, l->block_numel * N, "gathered", 0);
  if (st != TIDE_OK) return st;
  const int64_t nin = rank < 0 ? (int64_t)N * P : P;
  for (int64_t i = 0; i < nin; ++i) {
    st = check_ptr(shards[i], l->shard_numel[i % P], "shards", i);
    if (st != TIDE_OK) return st;
  }
  const int64_t t0 = rank < 0 ? 0 : l->pk_rank_begin[rank];
  const int64_t t1 = rank < 0 ? (int64_t)l->pk_tiles.size() : l->pk_rank_begin[rank + 1];
  if (t1 <= t0) return TIDE_OK;
  st = ensure_device(l, stream);
  if (st != TIDE_OK) return st;

  const TableKey key = make_key(TIDE_OP_PACK, rank, (const void* const*)shards, (size_t)nin, nullptr, 0);
  PtrSlot* slot = nullptr;
  st = acquire_table(
      l, key, (size_t)N * P,
      [&](void** dst) {  // rank-major; the entries of ranks not packed stay null
        if (rank < 0) {
          std::memcpy(dst, shards, (size_t)N * P * sizeof(void*));
        } else {
          std::memset(dst, 0, (size_t)N * P * sizeof(void*));
          std::memcpy(dst + (size_t)rank * P, shards, (size_t)P * sizeof(void*));
        }
      },
      stream, &slot);
  if (st != TIDE_OK) return st;

  PackArgs a;
  a.tiles = l->d_pk_tiles + t0;
  a.num_tiles = t1 - t0;
  a.stab = (const float* const*)slot->d_table;
  a.buf = gathered;
  a.num_params = P;
  a.err = l->d_err;
  a.ext = extents_of(l);
  cudaError_t e = launch_pack(a, grid_of(l, t1 - t0, 0), l->mode == TIDE_MODE_CAPPED, l->num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pack kernel launch");
  return mark_used(l, slot, stream);
}

tide_status_t tide_rs_stage_bf16(tide_layout_t l, const uint16_t* const* grads, uint16_t* slot,
                                 cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t P = l->num_params;
  if (P > 0 && !grads) return set_error(TIDE_ERR_INVALID_ARG, "grads table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  tide_status_t st = check_ptr(slot, l->block_numel * l->num_ranks, "slot", 0);
  if (st != TIDE_OK) return st;
  for (int32_t p = 0; p < P; ++p) {
    st = check_ptr(grads[p], l->d0[p] * l->inner[p], "grads", p);
    if (st != TIDE_OK) return st;
  }
  if (l->ag_tiles.empty()) return TIDE_OK;
  st = ensure_device(l, stream);
  if (st != TIDE_OK) return st;
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return copy_engine(l, slot, const_cast<uint16_t* const*>(grads), true, stream);

  const TableKey key = make_key(TIDE_OP_STAGE, 0, (const void* const*)grads, (size_t)P, nullptr, 0);
  PtrSlot* ps = nullptr;
  st = acquire_table(
      l, key, (size_t)P, [&](void** dst) { std::memcpy(dst, grads, (size_t)P * sizeof(void*)); }, stream,
      &ps);
  if (st != TIDE_OK) return st;
  AgArgs a;
  a.tiles = l->d_ag_tiles;
  a.num_tiles = (int64_t)l->ag_tiles.size();
  a.buf = slot;
  a.ptab = (uint16_t* const*)ps->d_table;
  cudaError_t e = launch_copy(l, a, true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "staging kernel launch");
  return mark_used(l, ps, stream);
}

tide_status_t tide_rs_staged_bf16_to_fp32(tide_layout_t l, const uint16_t* const* slots,
                                          float* const* shards, float scale, cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t N = l->num_ranks, P = l->num_params;
  if (P > 0 && (!slots || !shards)) return set_error(TIDE_ERR_INVALID_ARG, "pointer table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "reduce-scatter has no copy-engine mode");
  if (l->st_tiles.empty()) return TIDE_OK;
  for (int32_t k = 0; k < N; ++k) {
    tide_status_t st = check_ptr(slots[k], l->block_numel * N, "slots", k);
    if (st != TIDE_OK) return st;
  }
  for (int64_t i = 0, p = 0; i < (int64_t)N * P; ++i, p = (p + 1 == P ? 0 : p + 1)) {
    tide_status_t st = check_ptr(shards[i], l->shard_numel[p], "shards", i);
    if (st != TIDE_OK) return st;
  }
  // the kernel's per-parameter source table points every parameter at the
  // slot bases; the staged tiles carry slot offsets r*S + o_p + s
  const TableKey key = make_key(TIDE_OP_STAGED_RS, 0, (const void* const*)slots, (size_t)N,
                                (const void* const*)shards, (size_t)N * P);
  return run_rs(
      l, true, 0, (int64_t)l->st_tiles.size(), key,
      [&](void** dst) {
        for (int32_t p = 0; p < P; ++p)
          for (int32_t k = 0; k < N; ++k) dst[(size_t)p * N + k] = (void*)slots[k];
        std::memcpy(dst + (size_t)N * P, shards, (size_t)N * P * sizeof(void*));
      },
      scale, stream);
}

tide_status_t tide_layout_check_device(tide_layout_t l) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->device < 0) return TIDE_OK;  // nothing launched yet
  TIDE_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  int v = 0;
  TIDE_CUDA(cudaMemcpy(&v, l->d_err, sizeof v, cudaMemcpyDeviceToHost), "read of the error word");
  if (v == 0) return TIDE_OK;
  TIDE_CUDA(cudaMemset(l->d_err, 0, sizeof(int)), "reset of the error word");
  if (v & kDevErrRange)
    return set_error(TIDE_ERR_RANGE, std::string("a kernel of the debug build skipped a tile that addresses memory "
                                                 "outside its call's buffers") +
                                         (v & kDevErrTimeout ? "; a bounded wait also ran out" : ""));
  return set_error(TIDE_ERR_TIMEOUT, "a bounded wait in a bulk-copy kernel ran out; its copies were abandoned");
}

tide_status_t tide_layout_set_test_stall(tide_layout_t l, int64_t ns) {
  if (!l || ns < 0) return set_error(TIDE_ERR_INVALID_ARG, "NULL layout or negative time");
  std::lock_guard<std::mutex> g(l->mu);
  l->test_stall_ns = ns;
  return TIDE_OK;
}

}  // extern "C"
