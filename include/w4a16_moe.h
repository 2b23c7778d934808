/*
 * w4a16_moe.h -- C ABI of the GB300 (sm_103a) W4A16 mixture-of-experts expert path.
 *
 * The operation is the indexed W4A16 MoE expert GEMM described on
 * "vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x": BF16 activations,
 * uint4 weights with one BF16 scale per 32 consecutive K elements of each
 * output row (TL;DR; "vLLM integration": uint4, group-32, BF16 scales), and
 * tokens routed through sorted_ids / expert_ids / num_tokens_padded built by a
 * moe_align step ("Two kernel families": the indexed family consumes that
 * routing; "vLLM integration": over-allocated buffers, no host read-back of
 * the routed count, CUDA-graph capturable).  A layer is gate_up, SiLU-and-mul,
 * down and the top-k-weighted sum ("Measurements": per-layer time is gate_up
 * plus down; "humans& Beats FlashInfer's Best MoE Kernel by 25% on Blackwell
 * GPUs", "Dedicated warps keep the pipeline busy": FC1, FC2, top-K merge).
 *
 * Conventions shared by every call below
 *  - Every pointer named "device" is device memory owned by the caller; the
 *    library never allocates, frees or keeps a pointer after a call returns.
 *    Host pointers are read during the call only.
 *  - BF16 data is passed as uint16_t bit patterns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  No call synchronises the host or reads device memory back, so
 *    every call can be captured into a CUDA graph.
 *  - Every call returns a w4a16_status_t.  Argument errors are detected on the
 *    host before anything is enqueued; W4A16_CUDA_ERROR means a launch failed
 *    (the CUDA error is cleared and its text is kept for
 *    w4a16_last_error_detail()).
 *  - Problems found while kernels run (bad expert ids with validation on,
 *    a bounded wait that gave up, a packed-weight header mismatch) set bits in
 *    an optional caller-provided device int32 (`dev_err`, may be NULL); the
 *    host reads it when it chooses.  Kernels never trap.
 *  - Requires a GPU of compute capability 10.3 (sm_103a).
 */
#ifndef W4A16_MOE_H_
#define W4A16_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* w4a16_stream_t; /* identical to cudaStream_t */

typedef enum {
  W4A16_OK = 0,
  W4A16_INVALID_ARG = 1,         /* null pointer, negative or inconsistent size */
  W4A16_UNSUPPORTED = 2,         /* group != 32, K % 64, N % 128, block_m not in {16,32,64,128}, not sm_103 */
  W4A16_BAD_PACKED_WEIGHT = 3,   /* packed-weight descriptor magic/version/shape/mode mismatch */
  W4A16_WORKSPACE_TOO_SMALL = 4, /* workspace smaller than the matching *_workspace_size() */
  W4A16_CUDA_ERROR = 5           /* a CUDA launch or attribute call failed */
} w4a16_status_t;

/* Device error bits written (OR-ed) into `dev_err` by the kernels. */
#define W4A16_DEVERR_BAD_EXPERT_ID 0x1 /* an id outside [-1, E) was seen (treated as dropped) */
#define W4A16_DEVERR_CAPACITY 0x2      /* padded rows exceeded capacity (extra rows dropped) */
#define W4A16_DEVERR_TIMEOUT 0x4       /* a bounded pipeline wait gave up; output incomplete */
#define W4A16_DEVERR_BAD_HEADER 0x8    /* the packed blob's device header does not match */

/* Static text for a status code. */
const char* w4a16_status_string(w4a16_status_t status);
/* Text of the last failure seen by this host thread (empty if none). */
const char* w4a16_last_error_detail(void);

/* ------------------------------------------------------------------------------------------
 * Routing alignment ("Two kernel families"; "vLLM integration").
 *
 * topk_ids   device int32 [T, top_k], row-major; a local expert id in [0, E) or -1 for a
 *            dropped slot (an expert on another rank).  With validate != 0, any other value
 *            sets W4A16_DEVERR_BAD_EXPERT_ID in *dev_err; it is always treated as dropped.
 * Outputs (device, int32): sorted_ids [capacity], expert_ids [capacity / block_m],
 *            num_tokens_padded [1].
 * Result: the flat slot index i = t*top_k + s, stably sorted by expert (ascending i within an
 * expert), each expert's run padded up to a multiple of block_m with the sentinel T*top_k;
 * positions in [num_tokens_padded, capacity) also hold the sentinel.  expert_ids[b] is the
 * expert of rows [b*block_m, (b+1)*block_m) for b < num_tokens_padded / block_m and -1 after.
 * Experts with no routed slot get no block.  capacity must be a multiple of block_m and at
 * least w4a16_align_capacity(); 1 <= E <= 1024; T*top_k < 2^31.
 * ---------------------------------------------------------------------------------------- */
int64_t w4a16_align_capacity(int T, int top_k, int E, int block_m);
w4a16_status_t w4a16_moe_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                               int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* num_tokens_padded, int64_t capacity, int validate,
                               int32_t* dev_err, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Offline weight repack ("Grouped SM90 kernels": weights are packed once, the layout mode is
 * recorded in the prepared weight and checked at dispatch so a mismatch fails loudly).
 *
 * qweight  device int32 [E, N, K/8]: uint4 codes, element k in word k/8 at bits 4*(k%8)..+3
 *          (low nibble first); dequantised value (q - 8) * s.
 * scales   device uint16 (BF16) [E, N, K/32]: scale of elements [32g, 32g+32) of a row.
 * flags    W4A16_PACK_GATE_UP_PAIRED: N = 2*I holds gate rows [0, I) then up rows [I, 2I)
 *          (I % 64 == 0); every 128-row tile then carries 64 gate and the matching 64 up rows,
 *          which lets the GEMM fuse SiLU-and-mul.  0: plain row order.
 * packed   device buffer of w4a16_packed_bytes() bytes, 256-byte aligned; receives a device
 *          header and the tile stream.  `desc` (host) is filled on success and is what the
 *          GEMM calls take.  Requires group == 32, K % 64 == 0, N % 128 == 0.
 * Layout of the tile stream: for expert e, 128-row tile j, 64-wide K block kb, one 4608-byte
 * chunk (codes of 128 rows x 64 K, nibble-interleaved for pairwise BF16 conversion, then the
 * 128 x 2 scales); chunks of one (e, j) are contiguous along K.  After the chunks, one mode
 * byte per (e, j), padded to 16 bytes: a tile whose scales all lie in (0, 2^-5) stores them
 * as s * 2^133 and is converted with one fused multiply-add per pair of weights; any other
 * tile keeps its scales and the subtract-then-multiply conversion.  Both give the same BF16
 * weight, bf16_rne((q - 8) * s).
 * ---------------------------------------------------------------------------------------- */
#define W4A16_PACK_GATE_UP_PAIRED 0x1u
#define W4A16_PACK_NVFP4 0x2u /* set by w4a16_pack_weights_nvfp4: the blob holds NVFP4 weights */
#define W4A16_PACK_MAGIC 0x3631413457454f4dull /* "MOEW4A16" in little-endian bytes */
#define W4A16_PACK_VERSION 2u

typedef struct {
  uint64_t magic;   /* W4A16_PACK_MAGIC once filled */
  uint32_t version; /* W4A16_PACK_VERSION */
  uint32_t flags;   /* W4A16_PACK_* */
  int32_t E, N, K, group;
  uint64_t bytes;   /* size of the device blob */
  const void* data; /* device pointer to the blob (header + tiles) */
} w4a16_packed_weights_t;

size_t w4a16_packed_bytes(int E, int N, int K, int group, uint32_t flags);
w4a16_status_t w4a16_pack_weights(const int32_t* qweight, const uint16_t* scales, int E, int N,
                                  int K, int group, uint32_t flags, void* packed,
                                  size_t packed_bytes, w4a16_packed_weights_t* desc,
                                  w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * NVFP4 weights ("humans& Beats FlashInfer's Best MoE Kernel by 25% on Blackwell GPUs", "BF16
 * preserves each local product" and "Dedicated warps keep the pipeline busy"): blocks of 16
 * E2M1 values along K share one E4M3 scale; the weight is their product, which BF16 holds
 * exactly, so every GEMM and layer call runs unchanged on an NVFP4 blob (the descriptor's
 * W4A16_PACK_NVFP4 flag selects the conversion; activations stay BF16).
 *
 * codes   device uint8 [E, N, K/2]: element k of a row in byte k/2, low nibble for even k;
 *         E2M1 = sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * scales  device uint8 [E, N, K/16]: E4M3 (finite variant, bias 7) of elements [16g, 16g+16).
 * flags   0 or W4A16_PACK_GATE_UP_PAIRED (as above); the blob size is
 *         w4a16_packed_bytes(E, N, K, 16, W4A16_PACK_NVFP4 | flags), the same as for INT4.
 * A per-tensor FP32 second-level scale, where a checkpoint has one, is not part of this call
 * (the pages do not use one): fold it into the activations or the consumer of the output.
 * ---------------------------------------------------------------------------------------- */
w4a16_status_t w4a16_pack_weights_nvfp4(const uint8_t* codes, const uint8_t* scales, int E, int N,
                                        int K, uint32_t flags, void* packed, size_t packed_bytes,
                                        w4a16_packed_weights_t* desc, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Indexed grouped GEMM ("Two kernel families"; "H200 and Blackwell indexed decode").
 *
 * For every sorted position p < *num_tokens_padded with slot i = sorted_ids[p] < total_slots
 * and expert e = expert_ids[p / block_m]:
 *     C[row_c(p), :] = A[row_a(p), :] . dequant(W[e])^T      (FP32 accumulation, BF16 out)
 * row_a(p) = i / a_row_div (top_k for gate_up, 1 for down), or p with W4A16_A_ROWS_SORTED;
 * row_c(p) = i, or p with W4A16_C_ROWS_SORTED (then padding rows p are written too, as
 * zeros).  Rows of C not named are left untouched.  With W4A16_C_FP32 (epilogue NONE only)
 * C holds the FP32 sums unrounded (float, row stride ldc elements).
 * A  device BF16 [rows, K] with row stride lda elements (lda % 8 == 0, 16-byte aligned rows).
 * C  device BF16 (16-byte aligned, ldc % 8 == 0; FP32: ldc % 4 == 0) with row stride ldc
 *    elements; N columns (epilogue NONE) or N/2 columns
 *    (epilogue SILU_MUL: C[., j] = bf16(silu(g) * u), g and u the unrounded FP32 gate and up
 *    sums; needs a W4A16_PACK_GATE_UP_PAIRED weight).
 * workspace  device scratch of w4a16_gemm_workspace_size() bytes, 256-byte aligned; its
 *    counter words must be zero before the first use (w4a16_workspace_clear, or cudaMemset)
 *    and every call leaves them zero.  Concurrent calls must not share a workspace.
 * expected_rows_per_expert  host hint for the schedule (0: total_slots / E); it never
 *    changes results, which are independent of the schedule up to FP32 summation order
 *    (and bitwise identical between runs of the same schedule).
 * Schedule (picked per call unless `schedule` fixes it):
 *    - 16- and 32-token blocks: the K split of a tile is picked on the device from
 *      *num_tokens_padded.  When the routed (block, 128-row tile) units fill less than half
 *      the CTAs every tile is sliced, otherwise only the tiles of a last, partial wave (at
 *      most 8 slices of at least 1536 K elements each).  The slices' FP32 partials are summed
 *      in slice order by the last CTA to finish the tile (deterministic).  Without a
 *      workspace large enough for the partials tiles are never split.
 *    - K <= 512 at 16- and 32-token blocks: 2 or 4 consecutive tiles of a block share one
 *      work unit and its activation stages (tile groups).
 *    - 128-token blocks of sorted rows with at most 4 tiles (N <= 512) and K >= 4096: CTA
 *      pairs, one M = 256 MMA over the two CTAs of a cluster, each loading half the rows.
 * ---------------------------------------------------------------------------------------- */
#define W4A16_EPILOGUE_NONE 0
#define W4A16_EPILOGUE_SILU_MUL 1
#define W4A16_A_ROWS_SORTED 0x1u
#define W4A16_C_ROWS_SORTED 0x2u
#define W4A16_C_FP32 0x4u

typedef struct {
  const int32_t* sorted_ids;        /* device [capacity], 16-byte aligned */
  const int32_t* expert_ids;        /* device [capacity / block_m] */
  const int32_t* num_tokens_padded; /* device [1] */
  int64_t capacity;
  int32_t block_m;                  /* 16, 32, 64 or 128 */
  int32_t total_slots;              /* T * top_k, the sentinel value */
} w4a16_routing_t;

/* Schedule override, for measurements only (NULL or zeros: the planner decides). */
typedef struct {
  int32_t split_k;   /* K slices per tile (1..16) */
  int32_t num_ctas;  /* persistent CTAs */
  int32_t cta_pairs; /* 128-token blocks only: 1 = one CTA per MMA, 2 = CTA pairs (tcgen05
                        cta_group::2, M = 256 over two 128-row tiles; needs sorted activation
                        rows, an even tile count and no K split); 0 = planner */
  int32_t tile_group; /* 128-row weight tiles per work unit: 1 = one; 2 or 4 = consecutive
                         tiles of one block sharing its activation stages (16-token blocks up
                         to 4, 32-token blocks up to 2, K <= 512, no K split, N / 128 a
                         multiple); 0 = planner (the largest allowed) */
} w4a16_schedule_t;

size_t w4a16_gemm_workspace_size(int total_slots, int E, int N, int K, int block_m);
w4a16_status_t w4a16_workspace_clear(void* workspace, size_t workspace_bytes,
                                     w4a16_stream_t stream);
w4a16_status_t w4a16_moe_gemm(const uint16_t* A, int64_t lda, int a_row_div,
                              const w4a16_packed_weights_t* W, const w4a16_routing_t* routing,
                              int epilogue, uint32_t row_flags, uint16_t* C, int64_t ldc,
                              void* workspace, size_t workspace_bytes,
                              int expected_rows_per_expert, const w4a16_schedule_t* schedule,
                              int32_t* dev_err, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Activation rows in aligned order (the gather of "Two kernel families": indexed kernels read
 * token rows through sorted_ids).  out[p, :] = x[sorted_ids[p] / a_row_div, :] for every
 * routed position p < *num_tokens_padded; padding rows and rows past num_tokens_padded are
 * not written.  x device BF16 [rows, K] (row stride ldx), out device BF16 [capacity, K] (row
 * stride ldo); K % 8 == 0, ldx % 8 == 0, ldo % 8 == 0, both 16-byte aligned.  The result
 * feeds w4a16_moe_gemm with W4A16_A_ROWS_SORTED (activation tiles by 2-D TMA).
 * ---------------------------------------------------------------------------------------- */
w4a16_status_t w4a16_gather_rows(const uint16_t* x, int64_t ldx, int K, int a_row_div,
                                 const w4a16_routing_t* routing, uint16_t* out, int64_t ldo,
                                 w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Grouped contracts ("Grouped SM90 kernels": contiguous prefill and masked decode).  The page
 * builds these as a second kernel family with its own weight packers; here a small layout
 * kernel turns each layout into the aligned routing above and the indexed GEMM computes, so a
 * weight packed once by w4a16_pack_weights serves every contract (the gate/up pairing it
 * records is still checked: SiLU-and-mul needs a W4A16_PACK_GATE_UP_PAIRED weight).  Output
 * widths, alignment rules for A and C and the epilogues are those of w4a16_moe_gemm.
 *
 * Contiguous: A device BF16 [m, K] (row stride lda), rows concatenated by expert with each
 *   expert's group padded to a 128-row boundary (m % 128 == 0); m_indices device int32 [m],
 *   the expert of each row or -1 for padding.
 *     C[r, :] = A[r, :] . dequant(W[m_indices[r]])^T            for m_indices[r] >= 0.
 *   Padding rows of a 128-row block that holds valid rows are written as zeros; a block of
 *   padding only is left untouched.  A block whose valid ids differ, or an id outside [-1, E),
 *   sets W4A16_DEVERR_BAD_EXPERT_ID in *dev_err (when given); such a block is computed with
 *   the expert of its first valid row and out-of-range ids count as padding.
 * Masked: A device BF16 [G * max_m, K] (a [G, max_m, K] tensor is the same memory); masked_m
 *   device int32 [G], the valid rows of each expert (clamped to [0, max_m]; a value outside
 *   sets W4A16_DEVERR_CAPACITY); expected_m > 0 a host hint of rows per expert that selects
 *   the block size only; G must equal the weight's E (G <= 1024).
 *     C[g * max_m + r, :] = A[g * max_m + r, :] . dequant(W[g])^T  for r < masked_m[g];
 *   the other rows of C are left untouched (consumers ignore them).
 * workspace: device scratch of the matching *_workspace_size() bytes (it holds the routing),
 *   256-byte aligned, no initial contents required; concurrent calls must not share it.
 * Both are stream-ordered with no host synchronisation (graph capturable).
 * ---------------------------------------------------------------------------------------- */
size_t w4a16_contiguous_workspace_size(int64_t m);
w4a16_status_t w4a16_contiguous_gemm(const uint16_t* A, int64_t lda, int64_t m,
                                     const int32_t* m_indices, const w4a16_packed_weights_t* W,
                                     int epilogue, uint16_t* C, int64_t ldc, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err,
                                     w4a16_stream_t stream);
size_t w4a16_masked_workspace_size(int G, int max_m, int expected_m);
w4a16_status_t w4a16_masked_gemm(const uint16_t* A, int64_t lda, int G, int max_m,
                                 const int32_t* masked_m, int expected_m,
                                 const w4a16_packed_weights_t* W, int epilogue, uint16_t* C,
                                 int64_t ldc, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_err, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Indexed GEMM that allocates nothing.  The paper has no counterpart: this entry point exists
 * for callers that cannot hand the library a workspace, such as an inference-engine plugin
 * whose enqueue hook receives only its input and output buffers, or a serving loop that must
 * not call cudaMalloc after start-up (the call can synchronise the device and fragment memory
 * budgeted up front).
 *
 * Same arguments and results as w4a16_moe_gemm without the workspace: the K-split scratch
 * (arrival counters and FP32 partial sums) is a library-owned device array of
 * W4A16_STATIC_SCRATCH_BYTES that every GPU loading the library keeps until the process
 * exits.  The first call on a device looks up that array's device address (once per device,
 * with the device current); make that first call before any stream capture.  The address
 * belongs to the device's CUDA context: after a device reset the next call looks it up again
 * in the new context (so make that call before any capture too).  Each call
 * clears the counter words it needs with an asynchronous memset on `stream` and calls no
 * cudaMalloc, cudaFree or other allocating routine.  All calls share the one array: calls
 * whose kernels may overlap on the GPU (different streams, or concurrent host threads) race
 * on it and must be serialised by the caller.  A problem that would need more scratch than
 * the array holds is rejected with W4A16_WORKSPACE_TOO_SMALL.
 * ---------------------------------------------------------------------------------------- */
#define W4A16_STATIC_SCRATCH_BYTES ((size_t)16 * 1024 * 1024 + 8192)
w4a16_status_t w4a16_moe_gemm_static_scratch(const uint16_t* A, int64_t lda, int a_row_div,
                                             const w4a16_packed_weights_t* W,
                                             const w4a16_routing_t* routing, int epilogue,
                                             uint32_t row_flags, uint16_t* C, int64_t ldc,
                                             int expected_rows_per_expert,
                                             const w4a16_schedule_t* schedule, int32_t* dev_err,
                                             w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Top-k weighted sum (the "top-K expert output merge" of the humans& page).
 * Y device FP32 [T*top_k, H] (the per-slot down outputs, unrounded); out[t, :] =
 * bf16(sum over s ascending with topk_ids[t,s] >= 0 of topk_weights[t,s] * Y[t*top_k + s, :]),
 * FP32 accumulation; rows of dropped slots are not read.  H % 8 == 0.
 * ---------------------------------------------------------------------------------------- */
w4a16_status_t w4a16_topk_sum(const float* Y, const int32_t* topk_ids,
                              const float* topk_weights, int T, int top_k, int H,
                              uint16_t* out, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Whole layer: align -> row gather -> gate_up (SiLU-and-mul fused) -> down -> top-k sum, five
 * kernels chained with programmatic dependent launch ("humans& ...", "Blackwell hides the conversion
 * work": FC2 starts its weight work before FC1 completes).
 * x  device BF16 [T, H]; w13 packed [E, 2I, H] with W4A16_PACK_GATE_UP_PAIRED; w2 packed
 * [E, H, I]; topk_ids / topk_weights device [T, top_k]; out device BF16 [T, H] (a token
 * with no local slot gets a zero row).  E_global: experts the router chose from (0 = E),
 * used only for the schedule.  block_m: 0 = planner.  workspace of
 * w4a16_layer_workspace_size(..) bytes with the same block_m argument; no zeroing needed.
 * ---------------------------------------------------------------------------------------- */
/* Layer options.  W4A16_LAYER_FUSED_TOPK: the down GEMM's epilogue multiplies each slot's row
 * by its top-k weight and adds it into an FP32 [T, H] token sum with atomic vector reductions
 * (the per-slot [T*top_k, H] rows are never written), and a last kernel rounds the sums to BF16
 * ("humans& ...", "Dedicated warps keep the pipeline busy": the top-K expert output merge in the
 * MoE kernel).  Six kernels instead of five: a zeroing kernel precedes the GEMMs.  The order in
 * which the slots' terms are added then varies from run to run, so results are within the
 * tolerance but not bitwise reproducible; without the flag the sum runs over slots in order
 * and is reproducible. */
#define W4A16_LAYER_FUSED_TOPK 0x1u
/* W4A16_LAYER_FUSED: gate_up and down run as ONE persistent kernel (the single-kernel layer
 * of the humans& page's "Dedicated warps keep the pipeline busy", here without token
 * dispatch), with the top-k merge of W4A16_LAYER_FUSED_TOPK in its down epilogue.  Units of
 * the down GEMM follow the gate_up units in every CTA's sequence; a down unit's activation
 * loads wait until all gate_up tiles of its block are stored (a per-block counter in the
 * workspace, bounded wait), while its weights stream from the start, so the down projection
 * overlaps the gate_up tail.  The launch is cooperative (all CTAs resident); a wait that runs
 * out sets W4A16_DEVERR_TIMEOUT.  The kernel also zeroes the FP32 token sums first and rounds
 * them into out last (grid-wide phase counts; the align kernel clears the counts each call).
 * Kernels: align, (row gather for block_m >= 64), the fused GEMM.  Not bitwise reproducible,
 * as for W4A16_LAYER_FUSED_TOPK; implies it. */
#define W4A16_LAYER_FUSED 0x2u
/* Test hook for the bounded-wait error path, with W4A16_LAYER_FUSED only: every down unit
 * waits for one more finished gate_up tile than its block has, with a limit of 2^20 cycles
 * (about half a millisecond) instead of about a second.  Every such wait runs out: the CTA
 * gives up its remaining units, drains its copies, frees its tensor memory and returns, and
 * W4A16_DEVERR_TIMEOUT is set in *dev_err.  The call itself returns W4A16_OK; out is
 * incomplete.  Not for production use. */
#define W4A16_LAYER_DEBUG_WAIT_TIMEOUT 0x80000000u
int w4a16_plan_block_m(int T, int top_k, int E, int E_global);
size_t w4a16_layer_workspace_size(int T, int top_k, int E, int E_global, int H, int I,
                                  int block_m);
w4a16_status_t w4a16_moe_layer(const uint16_t* x, const w4a16_packed_weights_t* w13,
                               const w4a16_packed_weights_t* w2, const int32_t* topk_ids,
                               const float* topk_weights, int T, int top_k, int E_global,
                               int block_m, uint16_t* out, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err, w4a16_stream_t stream);
w4a16_status_t w4a16_moe_layer_ex(const uint16_t* x, const w4a16_packed_weights_t* w13,
                                  const w4a16_packed_weights_t* w2, const int32_t* topk_ids,
                                  const float* topk_weights, int T, int top_k, int E_global,
                                  int block_m, uint32_t layer_flags, uint16_t* out,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                  w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Host planner (no device work; usable without a GPU): the schedule w4a16_moe_gemm would
 * pick for these sizes on a GPU with num_sms SMs.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t block_m;
  int32_t split_k;     /* most K slices per tile the device may pick (see w4a16_moe_gemm) */
  int32_t num_ctas;
  int32_t stages;      /* weight/activation ring depth in shared memory */
  int32_t est_units;   /* estimated (block, tile, split) work units */
  int32_t cta_pairs;   /* 2: CTA pairs (when the activation rows are sorted, as the layer's
                          128-token blocks are), 1: one CTA per 128-row tile */
} w4a16_plan_t;

w4a16_status_t w4a16_plan_gemm(int total_slots, int E, int N, int K, int block_m,
                               int expected_rows_per_expert, int num_sms, w4a16_plan_t* plan);

/* ------------------------------------------------------------------------------------------
 * Test hook: dequantise expert `expert` of a packed weight with the GEMM's own device
 * conversion routine, into canonical order out device BF16 [N, K].
 * ---------------------------------------------------------------------------------------- */
w4a16_status_t w4a16_debug_dequant(const w4a16_packed_weights_t* W, int expert, uint16_t* out,
                                   w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_MOE_H_ */
