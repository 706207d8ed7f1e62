/*
 * tide.h — C ABI of libtide.so: layout-aware reduce-scatter math and
 * all-gather placement for FSDP2-style per-parameter storage, on one GPU
 * (sm_103a), with N data-parallel ranks simulated by N input/output sets.
 *
 * What the operations are (sources cited by page title and section):
 *
 *  - "FSDP通信终局：TIDE零拷贝集合通信优化" §FSDP2通信开销的根源: FSDP2 keeps
 *    parameters and gradients as one tensor per parameter, while its
 *    collectives work on flat rank-major buffers (each rank's elements
 *    contiguous, rank blocks one after another).  The all-gather output
 *    therefore has to be copied into parameter storage and gradients packed
 *    into a full fp32 buffer.  Reduce-scatter: every rank holds a full
 *    buffer; afterwards each rank holds one reduced shard.
 *  - same page, §TIDE的设计思路: TIDE-RS consumes the per-parameter bf16
 *    gradients directly and reduces them into fp32 shards (a mixed-precision
 *    mode NCCL lacks); TIDE-AG delivers shards straight into parameter
 *    storage, folding the placement into the collective's addressing.
 *    Intra-node accumulation uses copy engines and short-lived CTAs.
 *
 * This library computes, on one GPU, the data path of both: the reduction
 * math of TIDE-RS written straight into each rank's padded fp32 dim-0 shard
 * of every parameter (no flat pack buffer), and the placement of a
 * rank-major bf16 buffer straight into per-parameter storage (no copy-out).
 *
 * Sharding (FSDP2's dim-0 rule; the pages do not spell it out): parameter p
 * of shape [d0, ...] is viewed as a row-major [d0, inner] matrix
 * (inner = product of the trailing dims, 1 for a 1-D tensor, and a 0-dim
 * scalar is [1]).  With c = ceil(d0 / N), rank r owns rows
 * [r*c, min((r+1)*c, d0)) and its shard is padded with zero rows to c rows
 * (c * inner elements).  Ranks past the end own no rows (all padding).
 *
 * Rank-major buffer: N blocks of S elements; inside each block parameter
 * p's shard starts at offset o_p, o_0 = 0,
 * o_{p+1} = roundup(o_p + c_p * inner_p, A), S = roundup(o_P, A), A the
 * alignment in elements (8 by default: every shard starts on 16 bytes).
 *
 * Conventions for every call:
 *  - All device pointers are addresses the device that is current when the
 *    layout is first used can load from / store to: device memory, or pinned
 *    host memory mapped into the device address space (on Grace systems the
 *    kernels then read inputs and write results over NVLink-C2C with no
 *    separate copy).  Tables of pointers are HOST arrays read only during
 *    the call.  The caller owns every device buffer
 *    and keeps it alive until the work enqueued on `stream` completes.
 *  - Compute calls are asynchronous with respect to the host and never
 *    synchronise the device; every copy they make is cudaMemcpyAsync from
 *    pinned staging on the caller's stream.  The first compute call of a
 *    layout allocates its device tables and uploads its tile lists on its
 *    stream (calls on other streams are ordered after that upload); the
 *    first call with a new set of pointers uploads that pointer table into
 *    one of 8 cached slots per layout, each allocated once at its largest
 *    size, so no call frees device memory before tide_layout_destroy.  The
 *    host waits in one case only: a new pointer set that finds all 8 slots
 *    holding other sets waits for the last kernel that read the least
 *    recently used one before overwriting it.  After one call on a stream,
 *    the same calls with the same pointers can be captured from that stream
 *    into a CUDA graph and replayed (tested for tide_rs_bf16_to_fp32 and
 *    tide_ag_place).  A layout's first compute call, and a pointer set used
 *    for the first time, are refused inside a capture
 *    (TIDE_ERR_UNSUPPORTED); the device table of a pointer set used inside a
 *    capture is kept unchanged for the layout's lifetime (at most 8 pointer
 *    sets per layout can be held that way), so destroy the layout only once
 *    such graphs are no longer replayed.
 *  - A failed CUDA call is reported through the status and cleared from the
 *    runtime's per-thread last error.
 *  - Next to compute kernels, either cap the CTAs (TIDE_MODE_CAPPED) or put
 *    the compute on a stream of higher priority than the collective's
 *    (cudaStreamCreateWithPriority): outside the capped mode every launch is
 *    one short-lived CTA per tile, so the block scheduler dispatches the
 *    compute kernel's pending CTAs first and the collective fills what it
 *    leaves.  A stream's default priority is already the lowest (the range
 *    is 0, the default, to -3 on GB300), so the collective needs no special
 *    stream; the compute's stream must be raised, which only the caller can
 *    do.  Measured on GB300
 *    beside a loop of bf16 8192^3 GEMMs over 0.3 s windows (power-capped
 *    clock; 70B- and MoE-shaped layers): equal priority +279% to +601%
 *    GEMM time, depending on how the launches are submitted; low priority
 *    +7.2% to +9.6% with the reduce-scatter moving 0.28-0.35 TB/s, about
 *    what 8 capped CTAs cost (+6.8% to +8.6%, 0.41-0.44 TB/s); capped
 *    16 / 32 / 64 CTAs +12-14% / +22-26% / +49-51%.
 *  - A layout may be used from several host threads (calls are serialised
 *    internally).  Calls on different streams that write the same output
 *    buffers race, as any two kernels would.
 *  - Errors: TIDE_ERR_INVALID_ARG for null / out-of-range / overflowing
 *    arguments, TIDE_ERR_MISALIGNED for a pointer that is not 16-byte
 *    aligned (a null pointer for a zero-size tensor is accepted),
 *    TIDE_ERR_UNSUPPORTED for a mode that an operation does not have,
 *    TIDE_ERR_CUDA when the CUDA runtime reports an error (the message is
 *    kept per host thread, see tide_last_error()).  On any error nothing is
 *    enqueued on the stream.  A bounded wait that runs out inside a
 *    TIDE_MODE_BULK kernel is reported later, by tide_layout_check_device.
 */
#ifndef TIDE_H
#define TIDE_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define TIDE_API __attribute__((visibility("default")))
#else
#define TIDE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TIDE_OK = 0,
  TIDE_ERR_INVALID_ARG = 1,
  TIDE_ERR_MISALIGNED = 2,
  TIDE_ERR_UNSUPPORTED = 3,
  TIDE_ERR_CUDA = 4,
  TIDE_ERR_TIMEOUT = 5, /* a bounded device wait ran out (tide_layout_check_device) */
  TIDE_ERR_OUT_OF_MEMORY = 6,
  TIDE_ERR_RANGE = 7    /* debug build: a kernel skipped an out-of-range tile (tide_layout_check_device) */
} tide_status_t;

typedef enum {
  /* Kernels launched over the whole GPU: one CTA per tile of the layout's
   * work list, handed out in list order by the block scheduler. */
  TIDE_MODE_UNCAPPED = 0,
  /* Persistent kernels with at most `cta_cap` CTAs looping over the tile
   * list: the short-lived-CTA budget of "TIDE的设计思路", trading bandwidth
   * for SM time left to concurrent compute.  Each CTA is 1024 threads wide
   * (an SM hosting one is lost to full-SM compute kernels anyway, so it
   * keeps a whole SM's loads in flight).  In a grid of at most half the
   * SMs every warp walks its own tiles (the reduce-scatter for N <= 64,
   * and the placement, staging and pack), so one SM moves about 110 GB/s
   * of reduce-scatter traffic at N = 8 on GB300; larger grids hand each
   * tile to a whole CTA (placement, staging, pack: two 512-thread groups).
   * Results are the same in every form. */
  TIDE_MODE_CAPPED = 1,
  /* Placement and Slot-Reuse staging through the copy engines
   * (cudaMemcpy2DAsync, no SM use), the copy-engine path of "TIDE的设计思路".
   * The reduce-scatter forms and the pack have no copy-engine form: they
   * return TIDE_ERR_UNSUPPORTED in this mode. */
  TIDE_MODE_COPY_ENGINE = 2,
  /* The TMA bulk-copy engine (cp.async.bulk, mbarriers, every wait bounded;
   * see tide_layout_check_device).  Placement and staging: global -> shared
   * -> global copies issued by one lane per CTA.  Reduce-scatter (all three
   * forms, N <= 512; larger N runs the load/store kernel): one 288-thread
   * CTA per SM whose producer warp stages the rank slices of each chunk in a
   * 192 KiB shared-memory ring of 64 KiB stages and whose 8 consumer warps
   * sum them in ascending rank order.  Up to 16 ranks (8 when capped) one
   * stage holds all N slices of a chunk (64 KiB / N each); above, a stage
   * holds 16 ranks' 4 KiB slices (8 ranks' 8 KiB when capped) and a chunk
   * spans consecutive stages, its partial sums kept in registers.  The
   * no-allocation reduce-scatter and the per-rank placement run the
   * load/store kernels in this mode.  The pack runs as in
   * TIDE_MODE_UNCAPPED.  cta_cap > 0 caps the grid at cta_cap CTAs (one per
   * SM), cta_cap = 0 uses every SM. */
  TIDE_MODE_BULK = 3
} tide_mode_t;

/* Operations, for the launch-shape and tile-list queries. */
typedef enum {
  TIDE_OP_RS = 0,
  TIDE_OP_AG = 1,
  TIDE_OP_PACK = 2,
  TIDE_OP_STAGE = 3,     /* Slot-Reuse staging (runs the placement list backwards) */
  TIDE_OP_STAGED_RS = 4  /* reduce-scatter from staged slots */
} tide_op_t;

/* Maximum simulated ranks per layout. */
#define TIDE_MAX_RANKS 4096

typedef struct tide_layout_s* tide_layout_t;

/*
 * Create the layout descriptor of `num_params` parameters sharded over
 * `num_ranks` ranks (host-only; no CUDA call is made).
 *   ndims[p]    number of dims of parameter p (0 = scalar, treated as [1]);
 *   dims_flat   all dims back to back (sum of ndims entries), each >= 0;
 *   num_ranks   1 .. TIDE_MAX_RANKS;
 *   out         receives the handle (owned by the caller, free with
 *               tide_layout_destroy).
 * Parameter order inside a rank block is the order given.  num_params == 0
 * gives an empty layout whose calls do nothing.  Alignment A = 8 elements.
 */
TIDE_API tide_status_t tide_layout_create(int32_t num_params, const int32_t* ndims,
                                 const int64_t* dims_flat, int32_t num_ranks,
                                 tide_layout_t* out);

/* As tide_layout_create with an explicit offset alignment `align_elems`
 * (1, 2, 4, 8, 16, ... elements; a power of two <= 4096).  With A < 8 rank
 * slices may start off 16 bytes; such tiles take a scalar path. */
TIDE_API tide_status_t tide_layout_create_ex(int32_t num_params, const int32_t* ndims,
                                    const int64_t* dims_flat, int32_t num_ranks,
                                    int64_t align_elems, tide_layout_t* out);

/* Free the layout and every host/device resource it owns.  Work already
 * enqueued that uses the layout's device tables must have completed.
 * Passing NULL does nothing. */
TIDE_API void tide_layout_destroy(tide_layout_t layout);

/* Queries (host-only).  Indices out of range give TIDE_ERR_INVALID_ARG. */
TIDE_API tide_status_t tide_layout_num_params(tide_layout_t layout, int32_t* num_params);
TIDE_API tide_status_t tide_layout_num_ranks(tide_layout_t layout, int32_t* num_ranks);
/* S: elements of one rank block of the gathered buffer (the buffer holds
 * num_ranks * S bf16 elements). */
TIDE_API tide_status_t tide_layout_rank_block_numel(tide_layout_t layout, int64_t* block_numel);
/* c_p * inner_p: elements of each fp32 shard of parameter p. */
TIDE_API tide_status_t tide_layout_shard_numel(tide_layout_t layout, int32_t p, int64_t* numel);
/* o_p: offset of parameter p's shard inside every rank block. */
TIDE_API tide_status_t tide_layout_param_offset(tide_layout_t layout, int32_t p, int64_t* offset);
/* Rows of parameter p that rank r really owns (the rest of its shard is padding). */
TIDE_API tide_status_t tide_layout_valid_rows(tide_layout_t layout, int32_t p, int32_t r, int64_t* rows);
/* c_p = ceil(d0_p / N). */
TIDE_API tide_status_t tide_layout_chunk_rows(tide_layout_t layout, int32_t p, int64_t* rows);

/* Select how the compute calls run (default TIDE_MODE_UNCAPPED).  cta_cap is
 * read in TIDE_MODE_CAPPED (>= 1) and TIDE_MODE_BULK (>= 0, 0 = no cap).
 * A new layout starts in the mode named by the environment variable
 * TIDE_MODE ("uncapped", "capped", "copy_engine" or "bulk", with the cap in
 * TIDE_CTA_CAP) when it is set to a valid choice.  TIDE_TILE_BYTES (4096 ..
 * 16777216) sets the bf16 bytes read per reduce-scatter tile (default 256
 * KiB) of layouts created afterwards. */
TIDE_API tide_status_t tide_layout_set_mode(tide_layout_t layout, tide_mode_t mode, int32_t cta_cap);

/* Current mode and CTA cap (host-only). */
TIDE_API tide_status_t tide_layout_get_mode(tide_layout_t layout, tide_mode_t* mode, int32_t* cta_cap);

/* Grid and block size the next launch of `op` will use under the current
 * mode, for the device that is current (grid 0 means no kernel: an empty
 * layout, or copy-engine placement).  Host-only until the first compute
 * call; uses the current device's SM count. */
TIDE_API tide_status_t tide_layout_launch_shape(tide_layout_t layout, tide_op_t op, int32_t* grid,
                                       int32_t* block);

/* Work list of `op` as rows of 6 int64 (param, rank, src_offset,
 * dst_offset, length, flags) into `rows` (capacity `cap` rows); *count gets
 * the number of tiles.  Host-only; for tests and tools. */
TIDE_API tide_status_t tide_layout_tiles(tide_layout_t layout, tide_op_t op, int64_t* rows, int64_t cap,
                                int64_t* count);

/*
 * Reduce-scatter math of TIDE-RS ("TIDE的设计思路"): for every rank r,
 * parameter p, shard row i' < c_p and column j, with i = r*c_p + i',
 *   shards[r*P + p][i'*inner_p + j] =
 *       scale * sum_{k=0}^{N-1} f32(grads[k*P + p][i*inner_p + j])   if i < d0_p
 *       +0.0f                                                       otherwise,
 * the sum taken in fp32 in ascending k from +0.0f, every add and the final
 * multiply rounded to nearest even, subnormals kept.
 *   grads   host array of N*P device pointers, rank-major: grads[k*P + p]
 *           is rank k's bf16 gradient of parameter p (d0_p*inner_p
 *           elements, contiguous row-major, 16-byte aligned);
 *   shards  host array of N*P device pointers: shards[r*P + p] is rank r's
 *           fp32 shard of parameter p (c_p*inner_p elements, 16-byte
 *           aligned); every element, padding included, is written;
 *   scale   applied after the sum (1/N averages);
 *   stream  CUDA stream the kernel is enqueued on.
 * Outputs must not overlap inputs or each other.  In TIDE_MODE_COPY_ENGINE
 * returns TIDE_ERR_UNSUPPORTED.
 */
TIDE_API tide_status_t tide_rs_bf16_to_fp32(tide_layout_t layout, const uint16_t* const* grads,
                                   float* const* shards, float scale, cudaStream_t stream);

/*
 * Placement of TIDE-AG ("TIDE的设计思路"; rank-major buffer of
 * "FSDP2通信开销的根源"): for every parameter p, row i < d0_p and column j,
 * with r = i / c_p,
 *   params[p][i*inner_p + j] = gathered[r*S + o_p + (i - r*c_p)*inner_p + j].
 * Padding and alignment slots of `gathered` are never read.
 *   gathered  device pointer to N*S bf16 elements (16-byte aligned);
 *   params    host array of P device pointers, params[p] is parameter p's
 *             bf16 storage (d0_p*inner_p elements, 16-byte aligned);
 *   stream    CUDA stream the work is enqueued on (a kernel, or copy-engine
 *             copies in TIDE_MODE_COPY_ENGINE).
 * A bit copy: the result is bit-exact.  Outputs must not overlap the input.
 */
TIDE_API tide_status_t tide_ag_place(tide_layout_t layout, const uint16_t* gathered,
                            uint16_t* const* params, cudaStream_t stream);

/*
 * Reduce-scatter output of ONE rank: what a single GPU of an FSDP2 job keeps
 * after the collective ("FSDP2通信开销的根源": each rank ends with one
 * reduced shard).  Same arithmetic as tide_rs_bf16_to_fp32, restricted to
 * rank `rank`:
 *   shards[p][i'*inner_p + j] = scale * sum_k f32(grads[k*P + p][(rank*c_p + i')*inner_p + j])
 * (+0.0f in padding rows), summed in ascending k from +0.0f.
 *   rank    0 .. N-1;
 *   grads   host array of N*P device pointers, as for tide_rs_bf16_to_fp32;
 *   shards  host array of P device pointers: that rank's fp32 shard of each
 *           parameter (c_p*inner_p elements, 16-byte aligned).
 * Reads N*(c_p rows) of every gradient instead of all rows.  Modes as for
 * tide_rs_bf16_to_fp32 (TIDE_ERR_UNSUPPORTED in TIDE_MODE_COPY_ENGINE).
 */
TIDE_API tide_status_t tide_rs_bf16_to_fp32_rank(tide_layout_t layout, int32_t rank,
                                                 const uint16_t* const* grads, float* const* shards,
                                                 float scale, cudaStream_t stream);

/*
 * Placement from per-rank buffers: TIDE-AG delivers each rank's shards
 * straight into parameter storage ("TIDE的设计思路").  With one process per
 * rank, rank r's packed block sits in rank r's own rank-major buffer; this
 * call reads every rank's block from that rank's buffer, so no all-gather
 * copy into a local buffer precedes the placement:
 *   params[p][i*inner_p + j] = gathered[r][r*S + o_p + (i - r*c_p)*inner_p + j],  r = i / c_p.
 * With gathered[k] all equal it is tide_ag_place.
 *   gathered  host array of N device pointers, each to a whole N*S bf16
 *             rank-major buffer (16-byte aligned; only block k of
 *             gathered[k] is read), e.g. peers' buffers from tide_ipc_open;
 *   params    host array of P device pointers, as for tide_ag_place.
 * Runs the load/store placement kernel in every mode but
 * TIDE_MODE_COPY_ENGINE (one cudaMemcpyAsync per parameter and rank).
 * Bit copy.
 */
TIDE_API tide_status_t tide_ag_place_ranks(tide_layout_t layout, const uint16_t* const* gathered,
                                           uint16_t* const* params, cudaStream_t stream);

/*
 * All-gather input pack: FSDP2 gathers each rank's padded shard in the bf16
 * parameter dtype, so after the optimizer step a rank casts its fp32 shard
 * to bf16 into its slot of the rank-major buffer ("FSDP2通信开销的根源"):
 *   gathered[r*S + o_p + e] = bf16_rne(shards_r[p][e])   for e < c_p*inner_p,
 * padding rows included; bf16_rne rounds to nearest, ties to even, keeps
 * NaN (quiet, sign and top payload kept) and rounds overflow to infinity.
 * Alignment gaps between shards are not written.
 *   rank      0 .. N-1: `shards` holds P device pointers (that rank's fp32
 *             shards) and only block `rank` is written;
 *             -1: `shards` holds N*P pointers (rank-major, as the output of
 *             tide_rs_bf16_to_fp32) and every block is written;
 *   gathered  device pointer to the N*S bf16 buffer (16-byte aligned).
 * TIDE_ERR_UNSUPPORTED in TIDE_MODE_COPY_ENGINE (a cast needs the SMs).
 */
TIDE_API tide_status_t tide_ag_pack_bf16(tide_layout_t layout, int32_t rank, const float* const* shards,
                                         uint16_t* gathered, cudaStream_t stream);

/*
 * Slot-Reuse staging ("TIDE的设计思路": the optional Slot-Reuse mechanism
 * stages gradients in the vacated all-gather slot, and a two-stage pipeline
 * decouples gradient reads from the collective's progress).  Copies one
 * rank's per-parameter bf16 gradients into its slot, a buffer with the
 * rank-major layout of the gathered buffer, destination by destination:
 *   slot[r*S + o_p + e] = grads[p][r*c_p*inner_p + e]   for e < v_{p,r}*inner_p.
 * Padding and alignment slots are not written.  Every rank stages the same
 * way into its own slot.
 *   grads  host array of P device pointers (bf16, 16-byte aligned);
 *   slot   device pointer to N*S bf16 elements (16-byte aligned).
 * Bit copy.  In TIDE_MODE_COPY_ENGINE the copy runs on the copy engines
 * (the placement's 2-D copies reversed).
 */
TIDE_API tide_status_t tide_rs_stage_bf16(tide_layout_t layout, const uint16_t* const* grads, uint16_t* slot,
                                          cudaStream_t stream);

/*
 * Reduce-scatter from N staged slots (the second stage of the Slot-Reuse
 * pipeline): every rank's inputs are now one contiguous rank-major buffer.
 *   shards[r*P + p][e] = scale * sum_{k=0}^{N-1} f32(slots[k][r*S + o_p + e])  for e < v_{p,r}*inner_p,
 *   +0.0f in padding rows; fp32 sum in ascending k from +0.0f — bit for bit
 *   the result of tide_rs_bf16_to_fp32 on the unstaged gradients.
 *   slots   host array of N device pointers (N*S bf16 each, 16-byte aligned);
 *   shards  host array of N*P device pointers, as for tide_rs_bf16_to_fp32.
 * Padding slots of the slots are never read.  TIDE_ERR_UNSUPPORTED in
 * TIDE_MODE_COPY_ENGINE.
 */
TIDE_API tide_status_t tide_rs_staged_bf16_to_fp32(tide_layout_t layout, const uint16_t* const* slots,
                                                   float* const* shards, float scale, cudaStream_t stream);

/* Bytes of the device array behind tide_rs_bf16_to_fp32_noalloc. */
#define TIDE_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * Reduce-scatter that allocates nothing.  The pages have no counterpart: it
 * exists for callers that cannot call cudaMalloc — for example a framework
 * whose caching allocator owns all device memory and must not see
 * allocations it does not track, a process under a hard device-memory cap
 * with every byte reserved, or a step that cannot absorb the device-wide
 * synchronisation of a later cudaFree.  tide_rs_bf16_to_fp32 allocates its
 * device tile list and pointer tables on a layout's first call; this variant
 * never does, so together with the host-only tide_layout_create a caller can
 * run the reduce-scatter without any allocation.
 *
 * Same arguments, result (bit for bit) and modes as tide_rs_bf16_to_fp32
 * (in TIDE_MODE_BULK it runs the load/store kernel, one CTA per tile).
 * The kernel's scratch (the layout's tile list, 32 bytes per tile, plus
 * 2*N*P device pointers) is copied on `stream` into one file-scope device
 * array of TIDE_NOALLOC_SCRATCH_BYTES (4 MiB) that every GPU loading the
 * library holds until the process exits; a layout that needs more returns
 * TIDE_ERR_INVALID_ARG without enqueuing anything.  Every byte the kernel
 * reads from the array was written either by this call or by the last call
 * that copied into it, whose copies stream order puts ahead of this kernel,
 * so nothing has to start at zero.  All calls share the array, which keeps
 * the last call's tables: calls that overlap on the GPU (on different
 * streams, or from different layouts without stream ordering between them)
 * race.  The first call on each device, and the first after the device's
 * CUDA context was replaced (cudaDeviceReset), looks up the array's device
 * address (cudaGetSymbolAddress) and copies the tables again (every call
 * does, if the driver cannot report a context id).  The tables
 * are copied from pageable host memory, so a call that copies returns only
 * once the stream's earlier work has completed and the driver has taken
 * its copy of them; calls on one device are serialised with each other
 * (one lock per device) while they check, copy and launch, and calls on
 * different devices do not wait for each other.  A call on the same stream,
 * with the same layout and the same pointers as the call that last filled
 * the array, copies nothing and returns at once (stream order already puts
 * the earlier copies before its kernel).  Inside a stream capture the call
 * returns TIDE_ERR_UNSUPPORTED: pageable copies cannot be replayed from a
 * CUDA graph.  No cudaMalloc, cudaFree or other allocating routine is
 * called.
 */
TIDE_API tide_status_t tide_rs_bf16_to_fp32_noalloc(tide_layout_t layout, const uint16_t* const* grads,
                                                    float* const* shards, float scale,
                                                    cudaStream_t stream);

/*
 * Rank processes: peer memory.  With one process per rank, TIDE-RS reads
 * every rank's per-parameter bf16 gradients directly
 * ("FSDP通信终局：TIDE零拷贝集合通信优化" §TIDE的设计思路) and each rank keeps only
 * its own shard; the data a rank brings in from its peers is (N-1)/N of the
 * reduce-scatter input ("通信量分析" §带宽饱和和节点扩展).  These calls map a
 * peer's buffers into this process so that rank r runs
 * tide_rs_bf16_to_fp32_rank(r) with a pointer table whose entries for the
 * other ranks are their gradients, and reads its peers' packed blocks of
 * the rank-major buffer before tide_ag_place.  No multicast, no library
 * collective: the loads are the library's own kernels (keep such calls in
 * TIDE_MODE_UNCAPPED or TIDE_MODE_CAPPED: the TMA kernels of TIDE_MODE_BULK
 * are for this process's own memory).  Tested with every rank process on
 * one GPU; across GPUs the devices must have peer access.
 *
 *   tide_ipc_export: `handle` (TIDE_IPC_HANDLE_BYTES bytes) receives the IPC
 *     handle of the cudaMalloc allocation that contains device pointer
 *     `ptr`, `offset` the byte offset of `ptr` in it.  The allocation must
 *     stay alive until every peer has closed it.
 *   tide_ipc_open: maps the allocation of a peer's handle into this process
 *     (on the current device); `base` receives its address, to which the
 *     peer's offsets are added.  A handle is opened once per process.
 *   tide_ipc_close: unmaps a base returned by tide_ipc_open.
 * Errors: TIDE_ERR_INVALID_ARG (NULL, or a pointer outside any device
 * allocation), TIDE_ERR_CUDA (the CUDA IPC call failed).
 */
#define TIDE_IPC_HANDLE_BYTES 64
TIDE_API tide_status_t tide_ipc_export(const void* ptr, uint8_t* handle, uint64_t* offset);
TIDE_API tide_status_t tide_ipc_open(const uint8_t* handle, void** base);
TIDE_API tide_status_t tide_ipc_close(void* base);

/*
 * Device-side failure report.  Synchronises the device, then reads and clears
 * the layout's device error word: TIDE_ERR_TIMEOUT if, since the last check,
 * a bounded wait inside a bulk-copy (TMA engine) kernel of this layout ran
 * out — the kernel then abandoned its remaining copies, so the outputs of
 * that call are incomplete — else TIDE_OK.  The wait bound is 2 s.  In a
 * debug build (see tide_build_info) every kernel first checks each tile it
 * fetches against the extents of its call's buffers (the test
 * tide_layout_check_tiles applies); a tile that fails is skipped and this
 * call returns TIDE_ERR_RANGE (taking precedence over a timeout).  The
 * no-allocation entry point has no device error word and is not checked.
 */
TIDE_API tide_status_t tide_layout_check_device(tide_layout_t layout);

/*
 * Test hook for the bounded waits: with ns > 0, every following bulk-copy
 * launch of this layout waits on a barrier nothing arrives on, bounded by ns
 * nanoseconds, reports the timeout through the error word and copies
 * nothing; ns = 0 turns the hook off.  Lets tests exercise the timeout path
 * without faulting or hanging a GPU.
 */
TIDE_API tide_status_t tide_layout_set_test_stall(tide_layout_t layout, int64_t ns);

/*
 * Host check of a tile list against the layout's extents, with the test the
 * kernels of a debug build apply to every tile they fetch.  `rows` holds
 * `count` tiles of `op` as tide_layout_tiles writes them (6 int64: param,
 * rank, src_offset, dst_offset, length, flags).  A tile passes when its
 * parameter and rank exist, its offsets and length are non-negative, its
 * source run (unless it is a zero-fill tile) and its destination run lie
 * inside their buffers — the gradient / parameter storage of the parameter
 * (d0*inner elements), its fp32 shard (c*inner), or one rank-major buffer
 * (N*S) — its flags are known, zero-fill tiles appear only in reduce-scatter
 * lists, and a vector tile's offsets have the element alignment its 16-byte
 * accesses need.  *first_bad receives the index of the first failing tile,
 * or -1 when all pass.  Host-only.
 */
TIDE_API tide_status_t tide_layout_check_tiles(tide_layout_t layout, tide_op_t op, const int64_t* rows,
                                               int64_t count, int64_t* first_bad);

/* "release", or "debug: device range checks" for the library built with
 * TIDE_DEBUG=1 (libtide_debug.so). */
TIDE_API const char* tide_build_info(void);

/* Static description of a status code. */
TIDE_API const char* tide_status_string(tide_status_t status);

/* Message of the last failed call on this host thread ("" if none). */
TIDE_API const char* tide_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TIDE_H */
