/*
 * CPU oracle for the layout-aware reduce-scatter and all-gather placement.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call this code.  The
 * product library never links it, includes it or falls back to it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Plain, single-threaded, obviously correct C (built with -O2
 * -ffp-contract=off, no fast-math).  All loops follow the definitions below
 * with no blocking, fusion or reordering.
 *
 * Sources (web pages; cited by title and section):
 *  [TIDE]  "FSDP通信终局：TIDE零拷贝集合通信优化", sections
 *          "FSDP2通信开销的根源" (per-parameter storage vs. rank-major flat
 *          buffers; reduce-scatter semantics) and "TIDE的设计思路"
 *          (TIDE-RS consumes per-parameter bf16 gradients and reduces them to
 *          fp32 shards; TIDE-AG delivers shards straight into parameter
 *          storage).
 *  [VOL]   apxml "通信量分析", section "分片中的通信原语" (ReduceScatter averages
 *          gradients and leaves each GPU only the shard matching its
 *          parameter shard; AllGather rebuilds full parameters from shards).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *  - dim-0 sharding: FSDP2 splits each parameter along dim 0 into N chunks
 *    of c = ceil(d0 / N) rows, rank r owning rows [r*c, min((r+1)*c, d0)),
 *    padded with zero rows to c rows.
 *  - fp32 sum in ascending rank order, starting from +0.0f, then one fp32
 *    multiply by `scale`; IEEE round-to-nearest-even, subnormals kept.
 *  - rank-major buffer: rank r's block starts at r * S; inside a block,
 *    parameter p's shard starts at offset o_p, o_0 = 0,
 *    o_{p+1} = roundup(o_p + c_p * inner_p, A), S = roundup(o_P, A).
 *
 * Parity status: every function below is pinned by the CPU tests
 * (brute force, invariants, closed forms, an fp64 error bound, hand-derived
 * golden fixtures); none is "parity unpinned".
 */
#ifndef TIDE_ORACLE_H
#define TIDE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* c = ceil(d0 / N): rows of every rank's dim-0 chunk (0 when d0 == 0). */
int64_t oracle_chunk_rows(int64_t d0, int32_t num_ranks);

/* Valid (unpadded) rows of rank r: clamp(d0 - r * c, 0, c). */
int64_t oracle_valid_rows(int64_t d0, int32_t num_ranks, int32_t r);

/* Offsets o_p of each parameter's shard inside a rank block and the block
 * stride S, for alignment `align` (elements, >= 1).  Returns 0 on success. */
int oracle_layout(int32_t num_params, const int64_t* d0, const int64_t* inner, int32_t num_ranks,
                  int64_t align, int64_t* offsets, int64_t* block_numel);

/* One reduced element: fp32(sum_{k=0}^{N-1} f32(vals[k])) * scale, summed in
 * ascending k from +0.0f. */
float oracle_rs_element(int32_t num_ranks, const uint16_t* vals, float scale);

/* Reduce-scatter of bf16 per-parameter gradients into fp32 dim-0 shards.
 * grads[k * P + p]: rank k's gradient of parameter p, d0[p] * inner[p] bf16.
 * shards[r * P + p]: rank r's shard of parameter p, c_p * inner[p] fp32;
 * rows past d0[p] are written +0.0f.  Returns 0, or 1 without writing
 * anything when num_ranks is outside 1 .. 4096 (the size of the per-element
 * stack array of inputs). */
int oracle_rs(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
              const uint16_t* const* grads, float* const* shards, float scale);

/* Placement of a rank-major gathered bf16 buffer (num_ranks * block_numel
 * elements) into per-parameter storage params[p] (d0[p] * inner[p] bf16). */
void oracle_ag_place(int32_t num_ranks, int32_t num_params, const int64_t* d0,
                     const int64_t* inner, const int64_t* offsets, int64_t block_numel,
                     const uint16_t* gathered, uint16_t* const* params);

/* Index into the gathered buffer that parameter p's element (i, j) comes
 * from (used by sampled checks at sizes where a full placement is too slow). */
int64_t oracle_ag_source_index(int32_t num_ranks, int64_t d0, int64_t inner, int64_t offset,
                               int64_t block_numel, int64_t i, int64_t j);

/* Reduce-scatter output of one rank only: shards_r[p] (c_p * inner[p] fp32)
 * receives exactly what oracle_rs writes to shards[r * P + p].  Returns 0,
 * or 1 without writing anything when num_ranks is outside 1 .. 4096 or r is
 * not a rank. */
int oracle_rs_rank(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                   const uint16_t* const* grads, float* const* shards_r, float scale, int32_t r);

/* fp32 -> bf16 bits, round to nearest, ties to even; NaN keeps its sign and
 * top payload bits and becomes quiet; overflow rounds to infinity. */
uint16_t oracle_f32_to_bf16(float f);

/* All-gather input pack of rank r (FSDP2's cast of the fp32 shard to the
 * bf16 parameter dtype, written into the rank's block of the rank-major
 * buffer): gathered[r * S + o_p + e] = bf16(shards_r[p][e]) for every
 * e < c_p * inner[p], padding rows included.  Alignment gaps are untouched. */
void oracle_ag_pack(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                    const int64_t* offsets, int64_t block_numel, int32_t r,
                    const float* const* shards_r, uint16_t* gathered);

/* Slot-Reuse staging of rank k's gradients ([TIDE] "TIDE的设计思路": the
 * vacated all-gather slot holds the gradients): the slot has the rank-major
 * layout of the gathered buffer and receives, for every destination rank r,
 * the rows of each gradient that r owns:
 *   slot[r * S + o_p + e] = grad_k[p][r * c_p * inner[p] + e]  for e < v_{p,r} * inner[p].
 * Padding and alignment slots are untouched. */
void oracle_rs_stage(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                     const int64_t* offsets, int64_t block_numel, const uint16_t* const* grads_k,
                     uint16_t* slot);

/* Reduce-scatter from the N staged slots:
 *   shards[r * P + p][e] = scale * sum_{k=0}^{N-1} f32(slots[k][r * S + o_p + e])  for e < v_{p,r} * inner[p],
 *   +0.0f for the padding rows; fp32 sum in ascending k from +0.0f.
 * Returns 0, or 1 without writing anything when num_ranks is outside
 * 1 .. 4096. */
int oracle_rs_staged(int32_t num_ranks, int32_t num_params, const int64_t* d0, const int64_t* inner,
                     const int64_t* offsets, int64_t block_numel, const uint16_t* const* slots,
                     float* const* shards, float scale);

#ifdef __cplusplus
}
#endif

#endif /* TIDE_ORACLE_H */
