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
  int sms = 0, rs_occ = 0, ag_occ = 0;
};

tide_status_t query_device(const tide_layout_s* l, DeviceShape* d) {
  int dev = 0;
  TIDE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  TIDE_CUDA(cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev),
            "cudaDeviceGetAttribute(MultiProcessorCount)");
  TIDE_CUDA(rs_occupancy(l->num_ranks, &d->rs_occ), "occupancy of the reduce-scatter kernel");
  TIDE_CUDA(ag_occupancy(&d->ag_occ), "occupancy of the placement kernel");
  d->rs_occ = std::max(1, d->rs_occ);
  d->ag_occ = std::max(1, d->ag_occ);
  return TIDE_OK;
}

int grid_for(int64_t tiles, tide_mode_t mode, int32_t cap, int sms, int occ) {
  if (tiles <= 0) return 0;
  const int64_t g = mode == TIDE_MODE_CAPPED ? (int64_t)cap : (int64_t)sms * occ;
  return (int)std::min<int64_t>(tiles, g);
}

// Bind the layout to the current device on first use: query the SM count
// and occupancy, upload the tile lists.
tide_status_t ensure_device(tide_layout_s* l) {
  int dev = 0;
  TIDE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (l->device >= 0) {
    if (dev != l->device)
      return set_error(TIDE_ERR_INVALID_ARG, "layout is bound to device " + std::to_string(l->device) +
                                                 " but device " + std::to_string(dev) + " is current");
    return TIDE_OK;
  }
  DeviceShape d;
  tide_status_t st = query_device(l, &d);
  if (st != TIDE_OK) return st;
  TIDE_CUDA(cudaDeviceGetAttribute(&l->max_pitch, cudaDevAttrMaxPitch, dev),
            "cudaDeviceGetAttribute(MaxPitch)");
  const size_t rs_b = sizeof(Tile) * std::max<size_t>(1, l->rs_tiles.size());
  const size_t ag_b = sizeof(Tile) * std::max<size_t>(1, l->ag_tiles.size());
  TIDE_CUDA(cudaMalloc((void**)&l->d_rs_tiles, rs_b), "cudaMalloc(tile list)");
  TIDE_CUDA(cudaMalloc((void**)&l->d_ag_tiles, ag_b), "cudaMalloc(tile list)");
  if (!l->rs_tiles.empty())
    TIDE_CUDA(cudaMemcpy(l->d_rs_tiles, l->rs_tiles.data(), sizeof(Tile) * l->rs_tiles.size(),
                         cudaMemcpyHostToDevice),
              "upload of the reduce-scatter tile list");
  if (!l->ag_tiles.empty())
    TIDE_CUDA(cudaMemcpy(l->d_ag_tiles, l->ag_tiles.data(), sizeof(Tile) * l->ag_tiles.size(),
                         cudaMemcpyHostToDevice),
              "upload of the placement tile list");
  for (PtrSlot& s : l->slots) {
    TIDE_CUDA(cudaEventCreateWithFlags(&s.upload_ev, cudaEventDisableTiming), "cudaEventCreate");
    TIDE_CUDA(cudaEventCreateWithFlags(&s.use_ev, cudaEventDisableTiming), "cudaEventCreate");
  }
  l->num_sms = d.sms;
  l->rs_occ = d.rs_occ;
  l->ag_occ = d.ag_occ;
  l->device = dev;
  return TIDE_OK;
}

// Device copy of a pointer table, cached by content: steady-state training
// passes the same buffers every step, so a hit costs a key comparison and a
// stream-ordering wait.  `entries` is the table in device order.
tide_status_t acquire_table(tide_layout_s* l, std::vector<uintptr_t>& key,
                            const std::vector<void*>& entries, cudaStream_t stream, PtrSlot** out) {
  PtrSlot* hit = nullptr;
  for (PtrSlot& s : l->slots)
    if (s.used && s.key == key) {
      hit = &s;
      break;
    }
  if (hit) {
    if (hit->upload_stream != stream)
      TIDE_CUDA(cudaStreamWaitEvent(stream, hit->upload_ev, 0), "cudaStreamWaitEvent");
    *out = hit;
    return TIDE_OK;
  }
  PtrSlot* s = &l->slots[0];
  for (PtrSlot& c : l->slots) {
    if (!c.used) {
      s = &c;
      break;
    }
    if (c.last_use < s->last_use) s = &c;
  }
  // Kernels that read this slot's previous table, and its previous upload
  // from the staging buffer, must be done before either is overwritten.
  if (s->used) TIDE_CUDA(cudaEventSynchronize(s->use_ev), "cudaEventSynchronize");
  s->used = false;
  const size_t n = std::max<size_t>(1, entries.size());
  if (s->capacity < n) {
    if (s->d_table) cudaFree(s->d_table);
    if (s->h_staging) cudaFreeHost(s->h_staging);
    s->d_table = nullptr;
    s->h_staging = nullptr;
    s->capacity = 0;
    TIDE_CUDA(cudaMalloc((void**)&s->d_table, n * sizeof(void*)), "cudaMalloc(pointer table)");
    TIDE_CUDA(cudaMallocHost((void**)&s->h_staging, n * sizeof(void*)),
              "cudaMallocHost(pointer table staging)");
    s->capacity = n;
  }
  if (!entries.empty()) {
    std::memcpy(s->h_staging, entries.data(), entries.size() * sizeof(void*));
    TIDE_CUDA(cudaMemcpyAsync(s->d_table, s->h_staging, entries.size() * sizeof(void*),
                              cudaMemcpyHostToDevice, stream),
              "upload of the pointer table");
  }
  TIDE_CUDA(cudaEventRecord(s->upload_ev, stream), "cudaEventRecord");
  s->upload_stream = stream;
  s->key.swap(key);
  s->used = true;
  *out = s;
  return TIDE_OK;
}

tide_status_t mark_used(tide_layout_s* l, PtrSlot* s, cudaStream_t stream) {
  s->last_use = ++l->use_counter;
  TIDE_CUDA(cudaEventRecord(s->use_ev, stream), "cudaEventRecord");
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
// rank that owns a partial chunk.
tide_status_t ag_copy_engine(tide_layout_s* l, const uint16_t* buf, uint16_t* const* params,
                             cudaStream_t stream) {
  const int64_t S = l->block_numel;
  for (int32_t p = 0; p < l->num_params; ++p) {
    const int64_t c = l->chunk[p], inner = l->inner[p], d0 = l->d0[p];
    if (c == 0 || inner == 0) continue;
    const int64_t full = std::min<int64_t>(l->num_ranks, d0 / c);
    const size_t width = (size_t)(c * inner) * 2;
    const size_t spitch = (size_t)S * 2;
    if (full > 0) {
      if (spitch <= (size_t)l->max_pitch && full > 1) {
        TIDE_CUDA(cudaMemcpy2DAsync(params[p], width, buf + l->offset[p], spitch, width, (size_t)full,
                                    cudaMemcpyDeviceToDevice, stream),
                  "cudaMemcpy2DAsync");
      } else {
        for (int64_t r = 0; r < full; ++r)
          TIDE_CUDA(cudaMemcpyAsync(params[p] + r * c * inner, buf + r * S + l->offset[p], width,
                                    cudaMemcpyDeviceToDevice, stream),
                    "cudaMemcpyAsync");
      }
    }
    const int64_t rows = d0 - full * c;
    if (rows > 0 && full < l->num_ranks)
      TIDE_CUDA(cudaMemcpyAsync(params[p] + full * c * inner, buf + full * S + l->offset[p],
                                (size_t)(rows * inner) * 2, cudaMemcpyDeviceToDevice, stream),
                "cudaMemcpyAsync");
  }
  return TIDE_OK;
}

}  // namespace

int rs_grid(const tide_layout_s* l) {
  return grid_for((int64_t)l->rs_tiles.size(), l->mode, l->cta_cap, l->num_sms, l->rs_occ);
}

int ag_grid(const tide_layout_s* l) {
  return grid_for((int64_t)l->ag_tiles.size(), l->mode, l->cta_cap, l->num_sms, l->ag_occ);
}

}  // namespace tide

using namespace tide;

extern "C" {

void tide_layout_destroy(tide_layout_t l) {
  if (!l) return;
  if (l->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != l->device) cudaSetDevice(l->device);
    for (PtrSlot& s : l->slots) {
      if (s.use_ev && s.used) cudaEventSynchronize(s.use_ev);
      if (s.d_table) cudaFree(s.d_table);
      if (s.h_staging) cudaFreeHost(s.h_staging);
      if (s.upload_ev) cudaEventDestroy(s.upload_ev);
      if (s.use_ev) cudaEventDestroy(s.use_ev);
    }
    cudaFree(l->d_rs_tiles);
    cudaFree(l->d_ag_tiles);
    if (cur >= 0 && cur != l->device) cudaSetDevice(cur);
  }
  delete l;
}

tide_status_t tide_layout_launch_shape(tide_layout_t l, tide_op_t op, int32_t* grid, int32_t* block) {
  if (!l || !grid || !block) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  if (op != TIDE_OP_RS && op != TIDE_OP_AG) return set_error(TIDE_ERR_INVALID_ARG, "unknown op");
  std::lock_guard<std::mutex> g(l->mu);
  DeviceShape d;
  tide_status_t st = query_device(l, &d);
  if (st != TIDE_OK) return st;
  if (op == TIDE_OP_RS) {
    *grid = l->mode == TIDE_MODE_COPY_ENGINE
                ? 0
                : grid_for((int64_t)l->rs_tiles.size(), l->mode, l->cta_cap, d.sms, d.rs_occ);
    *block = rs_block(l->mode == TIDE_MODE_CAPPED);
  } else {
    *grid = l->mode == TIDE_MODE_COPY_ENGINE
                ? 0
                : grid_for((int64_t)l->ag_tiles.size(), l->mode, l->cta_cap, d.sms, d.ag_occ);
    *block = ag_block(l->mode == TIDE_MODE_CAPPED);
  }
  return TIDE_OK;
}

tide_status_t tide_rs_bf16_to_fp32(tide_layout_t l, const uint16_t* const* grads, float* const* shards,
                                   float scale, cudaStream_t stream) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "layout is NULL");
  const int32_t N = l->num_ranks, P = l->num_params;
  if (P > 0 && (!grads || !shards)) return set_error(TIDE_ERR_INVALID_ARG, "pointer table is NULL");
  std::lock_guard<std::mutex> g(l->mu);
  if (l->mode == TIDE_MODE_COPY_ENGINE)
    return set_error(TIDE_ERR_UNSUPPORTED, "reduce-scatter has no copy-engine mode");
  for (int64_t i = 0; i < (int64_t)N * P; ++i) {
    tide_status_t st = check_ptr(grads[i], l->d0[i % P] * l->inner[i % P], "grads", i);
    if (st == TIDE_OK) st = check_ptr(shards[i], l->shard_numel[i % P], "shards", i);
    if (st != TIDE_OK) return st;
  }
  if (l->rs_tiles.empty()) return TIDE_OK;
  tide_status_t st = ensure_device(l);
  if (st != TIDE_OK) return st;

  // device order: param-major gradient table, then rank-major shard table
  std::vector<uintptr_t> key;
  key.reserve(1 + 2 * (size_t)N * P);
  key.push_back((uintptr_t)TIDE_OP_RS);
  std::vector<void*> entries((size_t)2 * N * P);
  for (int32_t p = 0; p < P; ++p)
    for (int32_t k = 0; k < N; ++k) entries[(size_t)p * N + k] = (void*)grads[(size_t)k * P + p];
  for (int64_t i = 0; i < (int64_t)N * P; ++i) entries[(size_t)N * P + i] = (void*)shards[i];
  for (void* e : entries) key.push_back((uintptr_t)e);
  PtrSlot* slot = nullptr;
  st = acquire_table(l, key, entries, stream, &slot);
  if (st != TIDE_OK) return st;

  RsArgs a;
  a.tiles = l->d_rs_tiles;
  a.num_tiles = (int64_t)l->rs_tiles.size();
  a.gtab = (const uint16_t* const*)slot->d_table;
  a.stab = (float* const*)(slot->d_table + (size_t)N * P);
  a.num_ranks = N;
  a.num_params = P;
  a.scale = scale;
  cudaError_t e = launch_rs(a, rs_grid(l), l->mode == TIDE_MODE_CAPPED, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter kernel launch");
  return mark_used(l, slot, stream);
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
  st = ensure_device(l);
  if (st != TIDE_OK) return st;
  if (l->mode == TIDE_MODE_COPY_ENGINE) return ag_copy_engine(l, gathered, params, stream);

  std::vector<uintptr_t> key;
  key.reserve(1 + (size_t)P);
  key.push_back((uintptr_t)TIDE_OP_AG);
  std::vector<void*> entries((size_t)P);
  for (int32_t p = 0; p < P; ++p) {
    entries[p] = (void*)params[p];
    key.push_back((uintptr_t)params[p]);
  }
  PtrSlot* slot = nullptr;
  st = acquire_table(l, key, entries, stream, &slot);
  if (st != TIDE_OK) return st;

  AgArgs a;
  a.tiles = l->d_ag_tiles;
  a.num_tiles = (int64_t)l->ag_tiles.size();
  a.buf = gathered;
  a.ptab = (uint16_t* const*)slot->d_table;
  cudaError_t e = launch_ag(a, ag_grid(l), l->mode == TIDE_MODE_CAPPED, stream);
  if (e != cudaSuccess) return cuda_fail(e, "placement kernel launch");
  return mark_used(l, slot, stream);
}

}  // extern "C"
