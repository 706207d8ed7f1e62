// Host layout descriptor: per-parameter chunk / pad / offset tables and the
// tile work lists of the reduce-scatter and placement kernels.  Host-only:
// nothing here calls CUDA, so layouts can be built and inspected without a
// GPU.  Device copies are made lazily by tide_api.cpp.
//
// Sharding follows FSDP2's dim-0 rule (c = ceil(d0 / N) rows per rank,
// zero-padded); the rank-major block layout follows
// "FSDP通信终局：TIDE零拷贝集合通信优化" §FSDP2通信开销的根源.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>

#include "tide_internal.h"

namespace tide {

namespace {
thread_local std::string g_last_error;

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

int64_t roundup(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// bf16 bytes read per reduce-scatter tile: TIDE_RS_TILE_READ_BYTES, or the
// TIDE_TILE_BYTES environment variable (4 KiB .. 16 MiB) when set.
int64_t rs_tile_read_bytes() {
  const char* e = getenv("TIDE_TILE_BYTES");
  if (e && *e) {
    char* end = nullptr;
    const long long v = strtoll(e, &end, 10);
    if (end && *end == '\0' && v >= 4096 && v <= (16ll << 20)) return (int64_t)v;
  }
  return TIDE_RS_TILE_READ_BYTES;
}

// Elements per reduce-scatter tile: rs_tile_read_bytes() of bf16 reads across
// the N ranks, at least one full CTA pass (8 elements per thread).
int64_t rs_tile_elems(int32_t n) {
  int64_t t = rs_tile_read_bytes() / 2 / n;
  t = std::max<int64_t>(8 * TIDE_RS_THREADS, std::min<int64_t>(65536, t));
  return t / 8 * 8;
}
constexpr int64_t kAgTileElems = TIDE_AG_TILE_ELEMS;  // 32 KiB read + 32 KiB written: one CTA pass
constexpr int64_t kZeroTileElems = 65536;  // padding fill
// Small layouts: shrink tiles until a list has about this many (8 per SM of
// a 152-SM GPU), never below one pass of a reduce-scatter CTA (8 elements per
// thread), so small jobs still spread over the whole GPU.
constexpr int64_t kMinTiles = 1216;
constexpr int64_t kMinTileElems = 8 * TIDE_RS_THREADS;

int64_t fit_tile(int64_t t, int64_t total_elems) {
  const int64_t want = (total_elems + kMinTiles - 1) / kMinTiles;
  if (want >= t) return t;
  return std::max<int64_t>(kMinTileElems, (want + 7) / 8 * 8);
}

// Split [0, n) into near-equal runs of at most `t` elements, each run but
// the last a multiple of 8 elements.
template <typename F>
void split_runs(int64_t n, int64_t t, F&& emit) {
  if (n <= 0) return;
  const int64_t pieces = (n + t - 1) / t;
  const int64_t step = roundup((n + pieces - 1) / pieces, 8);
  for (int64_t s = 0; s < n; s += step) emit(s, std::min(step, n - s));
}

void build_tiles(tide_layout_s* l) {
  const int32_t N = l->num_ranks;
  int64_t total = 0;  // elements of every rank's padded shards
  for (int32_t p = 0; p < l->num_params; ++p) total += l->chunk[p] * l->inner[p] * N;
  const int64_t T = fit_tile(rs_tile_elems(N), total);
  const int64_t TA = fit_tile(kAgTileElems, total);
  l->rs_tiles.clear();
  l->ag_tiles.clear();
  l->pk_tiles.clear();
  l->st_tiles.clear();
  l->rs_rank_begin.assign(1, 0);
  l->pk_rank_begin.assign(1, 0);
  // rank-major: one rank's tiles are contiguous (single-rank calls launch a
  // sub-range of the list)
  for (int32_t r = 0; r < N; ++r) {
    for (int32_t p = 0; p < l->num_params; ++p) {
      const int64_t c = l->chunk[p], inner = l->inner[p], d0 = l->d0[p];
      const int64_t v = std::max<int64_t>(0, std::min<int64_t>(c, d0 - (int64_t)r * c));
      const int64_t seg = v * inner;
      const int64_t rs_src = (int64_t)r * c * inner;
      split_runs(seg, T, [&](int64_t s, int64_t n) {
        Tile t{rs_src + s, s, (int32_t)n, p, r, 0u};
        if (t.src % 8 == 0 && t.dst % 4 == 0) t.flags |= kTileVec;
        l->rs_tiles.push_back(t);
      });
      split_runs(c * inner - seg, kZeroTileElems, [&](int64_t s, int64_t n) {
        Tile t{0, seg + s, (int32_t)n, p, r, kTileZero};
        if (t.dst % 4 == 0) t.flags |= kTileVec;
        l->rs_tiles.push_back(t);
      });
      const int64_t ag_src = (int64_t)r * l->block_numel + l->offset[p];
      // staged reduce-scatter: the same runs read from every rank's slot at
      // r*S + o_p (padding runs as above)
      split_runs(seg, T, [&](int64_t s, int64_t n) {
        Tile t{ag_src + s, s, (int32_t)n, p, r, 0u};
        if (t.src % 8 == 0 && t.dst % 4 == 0) t.flags |= kTileVec;
        l->st_tiles.push_back(t);
      });
      split_runs(c * inner - seg, kZeroTileElems, [&](int64_t s, int64_t n) {
        Tile t{0, seg + s, (int32_t)n, p, r, kTileZero};
        if (t.dst % 4 == 0) t.flags |= kTileVec;
        l->st_tiles.push_back(t);
      });
      split_runs(seg, TA, [&](int64_t s, int64_t n) {
        Tile t{ag_src + s, rs_src + s, (int32_t)n, p, r, 0u};
        if (t.src % 8 == 0 && t.dst % 8 == 0) t.flags |= kTileVec;
        l->ag_tiles.push_back(t);
      });
      // pack: the whole padded shard (padding rows are part of the AG input)
      split_runs(c * inner, TA, [&](int64_t s, int64_t n) {
        Tile t{s, ag_src + s, (int32_t)n, p, r, 0u};
        if (t.src % 4 == 0 && t.dst % 8 == 0) t.flags |= kTileVec;
        l->pk_tiles.push_back(t);
      });
    }
    l->rs_rank_begin.push_back((int64_t)l->rs_tiles.size());
    l->pk_rank_begin.push_back((int64_t)l->pk_tiles.size());
  }
}

tide_status_t create(int32_t num_params, const int32_t* ndims, const int64_t* dims_flat,
                     int32_t num_ranks, int64_t align, tide_layout_t* out) {
  if (!out) return set_error(TIDE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_params < 0) return set_error(TIDE_ERR_INVALID_ARG, "num_params < 0");
  if (num_ranks < 1 || num_ranks > TIDE_MAX_RANKS)
    return set_error(TIDE_ERR_INVALID_ARG, "num_ranks out of range 1..TIDE_MAX_RANKS");
  if (align < 1 || align > 4096 || (align & (align - 1)))
    return set_error(TIDE_ERR_INVALID_ARG, "align_elems must be a power of two in 1..4096");
  if (num_params > 0 && !ndims) return set_error(TIDE_ERR_INVALID_ARG, "ndims is NULL");

  tide_layout_s* l = new (std::nothrow) tide_layout_s();
  if (!l) return set_error(TIDE_ERR_OUT_OF_MEMORY, "host allocation failed");
  static std::atomic<uint64_t> next_serial{1};
  l->serial = next_serial.fetch_add(1);
  l->num_ranks = num_ranks;
  l->num_params = num_params;
  l->align = align;
  int64_t pos = 0, o = 0, psi = 0;
  for (int32_t p = 0; p < num_params; ++p) {
    const int32_t nd = ndims[p];
    if (nd < 0 || nd > 64) {
      delete l;
      return set_error(TIDE_ERR_INVALID_ARG, "ndims[" + std::to_string(p) + "] out of range");
    }
    if (nd > 0 && !dims_flat) {
      delete l;
      return set_error(TIDE_ERR_INVALID_ARG, "dims_flat is NULL");
    }
    int64_t d0 = 1, inner = 1;
    for (int32_t d = 0; d < nd; ++d) {
      const int64_t v = dims_flat[pos + d];
      if (v < 0) {
        delete l;
        return set_error(TIDE_ERR_INVALID_ARG, "negative dim in parameter " + std::to_string(p));
      }
      if (d == 0) {
        d0 = v;
      } else if (!mul_ok(inner, v, &inner)) {
        delete l;
        return set_error(TIDE_ERR_INVALID_ARG, "size overflow in parameter " + std::to_string(p));
      }
    }
    pos += nd;
    int64_t numel = 0, shard = 0;
    const int64_t c = (d0 + num_ranks - 1) / num_ranks;
    if (!mul_ok(d0, inner, &numel) || !mul_ok(c, inner, &shard) || !add_ok(psi, numel, &psi) ||
        !add_ok(o, shard, &o) || o > INT64_MAX / 2 || numel > INT64_MAX / 8) {
      delete l;
      return set_error(TIDE_ERR_INVALID_ARG, "size overflow in parameter " + std::to_string(p));
    }
    l->d0.push_back(d0);
    l->inner.push_back(inner);
    l->chunk.push_back(c);
    l->shard_numel.push_back(shard);
    l->offset.push_back(o - shard);
    o = roundup(o, align);
  }
  l->block_numel = roundup(o, align);
  int64_t total = 0;
  if (!mul_ok(l->block_numel, num_ranks, &total) || total > INT64_MAX / 8) {
    delete l;
    return set_error(TIDE_ERR_INVALID_ARG, "gathered buffer size overflows");
  }
  try {
    build_tiles(l);
  } catch (const std::bad_alloc&) {
    delete l;
    return set_error(TIDE_ERR_OUT_OF_MEMORY, "host allocation of the tile lists failed");
  }
  // initial mode from the environment (TIDE_MODE, TIDE_CTA_CAP); anything
  // unrecognised leaves the default
  if (const char* m = getenv("TIDE_MODE")) {
    const char* c = getenv("TIDE_CTA_CAP");
    const long cap = c ? strtol(c, nullptr, 10) : 0;
    if (!strcmp(m, "uncapped")) {
      l->mode = TIDE_MODE_UNCAPPED;
    } else if (!strcmp(m, "capped") && cap >= 1 && cap <= (1l << 30)) {
      l->mode = TIDE_MODE_CAPPED;
      l->cta_cap = (int32_t)cap;
    } else if (!strcmp(m, "copy_engine")) {
      l->mode = TIDE_MODE_COPY_ENGINE;
    } else if (!strcmp(m, "bulk") && cap >= 0 && cap <= (1l << 30)) {
      l->mode = TIDE_MODE_BULK;
      l->cta_cap = (int32_t)cap;
    }
  }
  *out = l;
  return TIDE_OK;
}

}  // namespace

tide_status_t set_error(tide_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

tide_status_t cuda_fail(cudaError_t e, const char* what) {
  // the error is reported through the status; clear the runtime's per-thread
  // last error so it does not surface in the caller's next, unrelated check
  cudaGetLastError();
  std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return set_error(e == cudaErrorMemoryAllocation ? TIDE_ERR_OUT_OF_MEMORY : TIDE_ERR_CUDA, m);
}

}  // namespace tide

using tide::set_error;

extern "C" {

tide_status_t tide_layout_create(int32_t num_params, const int32_t* ndims, const int64_t* dims_flat,
                                 int32_t num_ranks, tide_layout_t* out) {
  return tide::create(num_params, ndims, dims_flat, num_ranks, 8, out);
}

tide_status_t tide_layout_create_ex(int32_t num_params, const int32_t* ndims,
                                    const int64_t* dims_flat, int32_t num_ranks,
                                    int64_t align_elems, tide_layout_t* out) {
  return tide::create(num_params, ndims, dims_flat, num_ranks, align_elems, out);
}

tide_status_t tide_layout_num_params(tide_layout_t l, int32_t* v) {
  if (!l || !v) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  *v = l->num_params;
  return TIDE_OK;
}

tide_status_t tide_layout_num_ranks(tide_layout_t l, int32_t* v) {
  if (!l || !v) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  *v = l->num_ranks;
  return TIDE_OK;
}

tide_status_t tide_layout_rank_block_numel(tide_layout_t l, int64_t* v) {
  if (!l || !v) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  *v = l->block_numel;
  return TIDE_OK;
}

#define TIDE_CHECK_P(l, p, v)                                                   \
  do {                                                                          \
    if (!(l) || !(v)) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");  \
    if ((p) < 0 || (p) >= (l)->num_params)                                      \
      return set_error(TIDE_ERR_INVALID_ARG, "parameter index out of range");   \
  } while (0)

tide_status_t tide_layout_shard_numel(tide_layout_t l, int32_t p, int64_t* v) {
  TIDE_CHECK_P(l, p, v);
  *v = l->shard_numel[p];
  return TIDE_OK;
}

tide_status_t tide_layout_param_offset(tide_layout_t l, int32_t p, int64_t* v) {
  TIDE_CHECK_P(l, p, v);
  *v = l->offset[p];
  return TIDE_OK;
}

tide_status_t tide_layout_chunk_rows(tide_layout_t l, int32_t p, int64_t* v) {
  TIDE_CHECK_P(l, p, v);
  *v = l->chunk[p];
  return TIDE_OK;
}

tide_status_t tide_layout_valid_rows(tide_layout_t l, int32_t p, int32_t r, int64_t* v) {
  TIDE_CHECK_P(l, p, v);
  if (r < 0 || r >= l->num_ranks) return set_error(TIDE_ERR_INVALID_ARG, "rank out of range");
  const int64_t c = l->chunk[p];
  *v = std::max<int64_t>(0, std::min<int64_t>(c, l->d0[p] - (int64_t)r * c));
  return TIDE_OK;
}

tide_status_t tide_layout_set_mode(tide_layout_t l, tide_mode_t mode, int32_t cta_cap) {
  if (!l) return set_error(TIDE_ERR_INVALID_ARG, "NULL layout");
  if (mode != TIDE_MODE_UNCAPPED && mode != TIDE_MODE_CAPPED && mode != TIDE_MODE_COPY_ENGINE &&
      mode != TIDE_MODE_BULK)
    return set_error(TIDE_ERR_INVALID_ARG, "unknown mode");
  if (mode == TIDE_MODE_CAPPED && cta_cap < 1)
    return set_error(TIDE_ERR_INVALID_ARG, "cta_cap must be >= 1 in TIDE_MODE_CAPPED");
  if (mode == TIDE_MODE_BULK && cta_cap < 0)
    return set_error(TIDE_ERR_INVALID_ARG, "cta_cap must be >= 0 in TIDE_MODE_BULK");
  std::lock_guard<std::mutex> g(l->mu);
  l->mode = mode;
  l->cta_cap = (mode == TIDE_MODE_CAPPED || mode == TIDE_MODE_BULK) ? cta_cap : 0;
  return TIDE_OK;
}

tide_status_t tide_layout_get_mode(tide_layout_t l, tide_mode_t* mode, int32_t* cta_cap) {
  if (!l || !mode || !cta_cap) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> g(l->mu);
  *mode = l->mode;
  *cta_cap = l->cta_cap;
  return TIDE_OK;
}

tide_status_t tide_layout_tiles(tide_layout_t l, tide_op_t op, int64_t* rows, int64_t cap,
                                int64_t* count) {
  if (!l || !count) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  if (op < TIDE_OP_RS || op > TIDE_OP_STAGED_RS) return set_error(TIDE_ERR_INVALID_ARG, "unknown op");
  const std::vector<tide::Tile>& t = op == TIDE_OP_RS     ? l->rs_tiles
                                     : op == TIDE_OP_PACK ? l->pk_tiles
                                     : op == TIDE_OP_STAGED_RS ? l->st_tiles
                                                               : l->ag_tiles;  // AG and STAGE
  *count = (int64_t)t.size();
  if (cap > 0 && !rows) return set_error(TIDE_ERR_INVALID_ARG, "rows is NULL");
  for (int64_t i = 0; i < std::min<int64_t>(cap, (int64_t)t.size()); ++i) {
    rows[6 * i + 0] = t[i].p;
    rows[6 * i + 1] = t[i].r;
    rows[6 * i + 2] = t[i].src;
    rows[6 * i + 3] = t[i].dst;
    rows[6 * i + 4] = t[i].len;
    rows[6 * i + 5] = t[i].flags;
  }
  return TIDE_OK;
}

tide_status_t tide_layout_check_tiles(tide_layout_t l, tide_op_t op, const int64_t* rows, int64_t count,
                                      int64_t* first_bad) {
  if (!l || !first_bad || count < 0 || (count > 0 && !rows))
    return set_error(TIDE_ERR_INVALID_ARG, "NULL argument or negative count");
  if (op < TIDE_OP_RS || op > TIDE_OP_STAGED_RS) return set_error(TIDE_ERR_INVALID_ARG, "unknown op");
  const int kind = op == TIDE_OP_RS          ? tide::kKindRs
                   : op == TIDE_OP_STAGED_RS ? tide::kKindStagedRs
                   : op == TIDE_OP_PACK      ? tide::kKindPack
                                             : tide::kKindCopy;  // placement and staging
  std::vector<int64_t> numel(l->num_params);
  for (int32_t p = 0; p < l->num_params; ++p) numel[p] = l->d0[p] * l->inner[p];
  tide::Extents e;
  e.grad_numel = numel.data();
  e.shard_numel = l->shard_numel.data();
  e.buf_numel = l->block_numel * l->num_ranks;
  e.num_params = l->num_params;
  e.num_ranks = l->num_ranks;
  *first_bad = -1;
  auto fits32 = [](int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; };
  for (int64_t i = 0; i < count; ++i) {
    const int64_t* r = rows + 6 * i;
    bool ok = fits32(r[0]) && fits32(r[1]) && fits32(r[4]) && r[5] >= 0 && r[5] <= (int64_t)UINT32_MAX;
    if (ok) {
      const tide::Tile t{r[2], r[3], (int32_t)r[4], (int32_t)r[0], (int32_t)r[1], (uint32_t)r[5]};
      ok = tide::tile_in_range(t, kind, e);
    }
    if (!ok) {
      *first_bad = i;
      break;
    }
  }
  return TIDE_OK;
}

const char* tide_build_info(void) { return TIDE_DEBUG ? "debug: device range checks" : "release"; }

const char* tide_status_string(tide_status_t s) {
  switch (s) {
    case TIDE_OK: return "TIDE_OK";
    case TIDE_ERR_INVALID_ARG: return "TIDE_ERR_INVALID_ARG: invalid argument";
    case TIDE_ERR_MISALIGNED: return "TIDE_ERR_MISALIGNED: pointer not 16-byte aligned";
    case TIDE_ERR_UNSUPPORTED: return "TIDE_ERR_UNSUPPORTED: operation not available in this mode";
    case TIDE_ERR_CUDA: return "TIDE_ERR_CUDA: CUDA runtime error";
    case TIDE_ERR_TIMEOUT: return "TIDE_ERR_TIMEOUT: bounded device wait expired";
    case TIDE_ERR_OUT_OF_MEMORY: return "TIDE_ERR_OUT_OF_MEMORY: allocation failed";
    case TIDE_ERR_RANGE: return "TIDE_ERR_RANGE: a debug-build kernel skipped an out-of-range tile";
  }
  return "unknown tide_status_t";
}

const char* tide_last_error(void) { return tide::g_last_error.c_str(); }

}  // extern "C"
