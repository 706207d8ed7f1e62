/*
 * CPU oracle for the layout-aware reduce-scatter and all-gather placement.
 * TEST INFRASTRUCTURE: see tide_oracle.h for who may call it, the sources it
 * follows and the readings it takes where the sources are silent.
 */
#include "tide_oracle.h"

#include <string.h>

/* Exact widening of a bf16 bit pattern to fp32: bf16 is the top half of an
 * fp32 word. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static int64_t roundup(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

/* Each reduced element gathers its N inputs into a stack array of this many
 * entries; the reduce-scatter functions refuse larger N before touching it. */
#define ORACLE_MAX_RANKS 4096

/* FSDP2 dim-0 chunking (reading: torch.chunk sizes padded to N chunks). */
int64_t oracle_chunk_rows(int64_t d0, int32_t num_ranks) {
  return (d0 + num_ranks - 1) / num_ranks;
}

int64_t oracle_valid_rows(int64_t d0, int32_t num_ranks, int32_t r) {
  int64_t c = oracle_chunk_rows(d0, num_ranks);
  int64_t v = d0 - (int64_t)r * c;
  if (v < 0) v = 0;
  if (v > c) v = c;
  return v;
}

/* Rank-major block layout ([TIDE] "FSDP2通信开销的根源": a rank's elements
 * are contiguous and the rank blocks follow one another). */
int oracle_layout(int32_t num_params, const int64_t* d0, const int64_t* inner, int32_t num_ranks,
                  int64_t align, int64_t* offsets, int64_t* block_numel) {
  if (num_params < 0 || num_ranks < 1 || align < 1) return 1;
  int64_t o = 0;
  for (int32_t p = 0; p < num_params; ++p) {
    offsets[p] = o;
    o = roundup(o + oracle_chunk_rows(d0[p], num_ranks) * inner[p], align);
  }
  *block_numel = roundup(o, align);
  return 0;
}

/* TIDE-RS arithmetic ([TIDE] "TIDE的设计思路": bf16 gradients in, fp32
 * shard out): the sum over ranks in fp32, ascending rank order, then the
 * scale. */
float oracle_rs_element(int32_t num_ranks, const uint16_t* vals, float scale) {
  float acc = 0.0f;
  for (int32_t k = 0; k < num_ranks; ++k) acc = acc + bf16_to_f32(vals[k]);
  return acc * scale;
}

/* Reduce-scatter ([TIDE] "FSDP2通信开销的根源"; [VOL] "分片中的通信原语"):
 * every rank holds a full gradient of each parameter; afterwards rank r holds
 * the reduced values of its own dim-0 chunk only. */
int oracle_rs(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
              const uint16_t* const* grads, float* const* shards, float scale) {
  uint16_t vals[ORACLE_MAX_RANKS];
  if (num_ranks < 1 || num_ranks > ORACLE_MAX_RANKS) return 1;
  for (int32_t p = 0; p < num_params; ++p) {
    const int64_t c = oracle_chunk_rows(d0[p], num_ranks);
    for (int32_t r = 0; r < num_ranks; ++r) {
      float* out = shards[(int64_t)r * num_params + p];
      for (int64_t ii = 0; ii < c; ++ii) {
        const int64_t i = (int64_t)r * c + ii; /* row of the full tensor */
        for (int64_t j = 0; j < inner[p]; ++j) {
          if (i < d0[p]) {
            for (int32_t k = 0; k < num_ranks; ++k)
              vals[k] = grads[(int64_t)k * num_params + p][i * inner[p] + j];
            out[ii * inner[p] + j] = oracle_rs_element(num_ranks, vals, scale);
          } else {
            out[ii * inner[p] + j] = 0.0f; /* padding row */
          }
        }
      }
    }
  }
  return 0;
}

int64_t oracle_ag_source_index(int32_t num_ranks, int64_t d0, int64_t inner, int64_t offset,
                               int64_t block_numel, int64_t i, int64_t j) {
  (void)d0;
  const int64_t c = oracle_chunk_rows(d0, num_ranks);
  const int64_t r = i / c; /* the rank whose chunk holds row i */
  return r * block_numel + offset + (i - r * c) * inner + j;
}

/* TIDE-AG placement ([TIDE] "TIDE的设计思路": shards go straight into the
 * parameter storage; "FSDP2通信开销的根源": the gathered buffer is rank-major). */
void oracle_ag_place(int32_t num_ranks, int32_t num_params, const int64_t* d0,
                     const int64_t* inner, const int64_t* offsets, int64_t block_numel,
                     const uint16_t* gathered, uint16_t* const* params) {
  for (int32_t p = 0; p < num_params; ++p)
    for (int64_t i = 0; i < d0[p]; ++i)
      for (int64_t j = 0; j < inner[p]; ++j)
        params[p][i * inner[p] + j] =
            gathered[oracle_ag_source_index(num_ranks, d0[p], inner[p], offsets[p], block_numel,
                                            i, j)];
}

int oracle_rs_rank(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                   const uint16_t* const* grads, float* const* shards_r, float scale, int32_t r) {
  uint16_t vals[ORACLE_MAX_RANKS];
  if (num_ranks < 1 || num_ranks > ORACLE_MAX_RANKS || r < 0 || r >= num_ranks) return 1;
  for (int32_t p = 0; p < num_params; ++p) {
    const int64_t c = oracle_chunk_rows(d0[p], num_ranks);
    for (int64_t ii = 0; ii < c; ++ii) {
      const int64_t i = (int64_t)r * c + ii;
      for (int64_t j = 0; j < inner[p]; ++j) {
        if (i < d0[p]) {
          for (int32_t k = 0; k < num_ranks; ++k)
            vals[k] = grads[(int64_t)k * num_params + p][i * inner[p] + j];
          shards_r[p][ii * inner[p] + j] = oracle_rs_element(num_ranks, vals, scale);
        } else {
          shards_r[p][ii * inner[p] + j] = 0.0f;
        }
      }
    }
  }
  return 0;
}

/* IEEE 754-2008 roundTiesToEven (§4.3.1) on the 16 bits dropped: adding
 * just under half a bf16 ulp (0x7FFF) plus the lowest kept bit carries into
 * the kept bits exactly when the dropped part exceeds half an ulp, or equals
 * it with an odd kept part; then truncate. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* FSDP2 all-gather input: the rank's padded shard in the parameter dtype,
 * at its place in the rank-major buffer ([TIDE] "FSDP2通信开销的根源"). */
void oracle_ag_pack(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                    const int64_t* offsets, int64_t block_numel, int32_t r,
                    const float* const* shards_r, uint16_t* gathered) {
  for (int32_t p = 0; p < num_params; ++p) {
    const int64_t n = oracle_chunk_rows(d0[p], num_ranks) * inner[p];
    for (int64_t e = 0; e < n; ++e)
      gathered[(int64_t)r * block_numel + offsets[p] + e] = oracle_f32_to_bf16(shards_r[p][e]);
  }
}

void oracle_rs_stage(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                     const int64_t* offsets, int64_t block_numel, const uint16_t* const* grads_k,
                     uint16_t* slot) {
  for (int32_t p = 0; p < num_params; ++p) {
    const int64_t c = oracle_chunk_rows(d0[p], num_ranks);
    for (int32_t r = 0; r < num_ranks; ++r) {
      const int64_t n = oracle_valid_rows(d0[p], num_ranks, r) * inner[p];
      for (int64_t e = 0; e < n; ++e)
        slot[(int64_t)r * block_numel + offsets[p] + e] = grads_k[p][(int64_t)r * c * inner[p] + e];
    }
  }
}

int oracle_rs_staged(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                     const int64_t* offsets, int64_t block_numel, const uint16_t* const* slots,
                     float* const* shards, float scale) {
  uint16_t vals[ORACLE_MAX_RANKS];
  if (num_ranks < 1 || num_ranks > ORACLE_MAX_RANKS) return 1;
  for (int32_t p = 0; p < num_params; ++p) {
    const int64_t c = oracle_chunk_rows(d0[p], num_ranks);
    for (int32_t r = 0; r < num_ranks; ++r) {
      float* out = shards[(int64_t)r * num_params + p];
      const int64_t n = oracle_valid_rows(d0[p], num_ranks, r) * inner[p];
      for (int64_t e = 0; e < c * inner[p]; ++e) {
        if (e < n) {
          for (int32_t k = 0; k < num_ranks; ++k)
            vals[k] = slots[k][(int64_t)r * block_numel + offsets[p] + e];
          out[e] = oracle_rs_element(num_ranks, vals, scale);
        } else {
          out[e] = 0.0f;
        }
      }
    }
  }
  return 0;
}
