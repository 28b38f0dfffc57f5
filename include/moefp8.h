/*
 * moefp8.h -- C ABI of libmoefp8.so: the block-FP8 mixture-of-experts layer forward on one
 * NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; the library keeps no pointer
 *   after the call returns and allocates no device memory on these paths (scratch space is the
 *   caller's `workspace`).  One exception: moe_blockfp8_forward also takes its activations
 *   (x, topk_ids, topk_w, out) in pinned host memory that the device reaches at the same
 *   address (moe_pointer_device_accessible); its kernels then read the inputs and write the
 *   output across the host link themselves, with no separate copy.
 * - Every call only enqueues work on `stream` and never synchronises it.  Routing metadata that
 *   the device produces (num_blocks, ...) stays on the device; the kernels read it there.
 * - Layouts are row-major and dense.  BF16 tensors are passed as `void*` (IEEE bfloat16 bit
 *   patterns), E4M3 tensors as `uint8_t*` (OCP e4m3fn codes).  Groups of 128 run along the
 *   contiguous (last) dimension.
 * - Return value: MOE_OK (0), or an error code with nothing enqueued.  A text explanation of the
 *   last error on the calling thread is available from moe_last_error_string().
 * - Errors that only the device can see (an expert map entry outside [-1, E_local), a bounded
 *   wait that ran out) set bits in a per-device status word read by moe_get_device_status();
 *   the affected items are skipped, never trapped.
 *
 * Names follow the pages that describe the method: lmdeploy PR #4956 "Perf/pytorch block fp8
 * moe decode", lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route preparation",
 * vLLM PR #53875 "Fuse clamped MoE activation and UE8M0 FP8 block quantization" and lmdeploy
 * PR #4228 "Moe Reduce kernel".
 */
#ifndef MOEFP8_H
#define MOEFP8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOEFP8_API __attribute__((visibility("default")))
#else
#define MOEFP8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = 1,          /* null or misaligned pointer, bad size, unsupported shape      */
    MOE_ERR_EXPERT_SLICE = 2, /* inconsistent local-expert slice (e.g. no map but E_local!=E) */
    MOE_ERR_UNSUPPORTED = 3,  /* no sm_103 device current, or the driver lacks an entry point */
    MOE_ERR_LAUNCH = 4,       /* a CUDA launch or tensor-map encode failed                   */
    MOE_ERR_WORKSPACE = 5     /* workspace null, misaligned (256 B) or smaller than required  */
} moe_status;

typedef enum { MOE_SCALE_F32 = 0, MOE_SCALE_UE8M0 = 1 } moe_scale_fmt;

/* IDENTITY: quantise the BF16 input as is (the MoE input hidden states).
 * SILU_MUL: a = bf16(SiLU(gate) * up), gate = first N columns, up = last N columns; a finite
 *           clamp_limit L clamps both halves to [-L, L] first.
 * SILU_MUL_GATE_UPPER: as SILU_MUL but the gate is clamped from above only (gate <= L). */
typedef enum { MOE_ACT_IDENTITY = 0, MOE_ACT_SILU_MUL = 1, MOE_ACT_SILU_MUL_GATE_UPPER = 2 } moe_act;

typedef enum { MOE_PROJ_GATE_UP = 0, MOE_PROJ_DOWN = 1 } moe_proj;
typedef enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype;
typedef enum { MOE_ROUTE_AUTO = 0, MOE_ROUTE_SINGLE_CTA = 1, MOE_ROUTE_MULTI_CTA = 2 } moe_route_path;
typedef enum { MOE_QUANT_AUTO = 0, MOE_QUANT_PER_GROUP = 1, MOE_QUANT_PERSISTENT = 2 } moe_quant_strategy;
/* ROW_MAJOR: [E_local, N_out, K] (K contiguous).  TILED: the same weights regrouped so that
 * every 128x128 block is one contiguous 16 KB run, ordered [E_local][N_out/128][K/128][128][128]
 * (see moe_blockfp8_pack_weights); the block scales keep their layout. */
typedef enum { MOE_WEIGHTS_ROW_MAJOR = 0, MOE_WEIGHTS_TILED = 1 } moe_weight_layout;
/* FUSED: route preparation, then one persistent kernel for everything else (see
 * moe_blockfp8_forward).  STAGED: one launch per stage through the same kernels as the per-stage
 * entry points.  STAGED_EPILOGUE_REDUCE: as STAGED, but the weighted top-k sum runs in the down
 * GEMM's epilogue instead of a separate reduce launch (block_m <= 32; with a larger block_m it
 * is STAGED).  AUTO: the path this library measured to be faster for the shape. */
typedef enum {
    MOE_FORWARD_AUTO = 0,
    MOE_FORWARD_FUSED = 1,
    MOE_FORWARD_STAGED = 2,
    MOE_FORWARD_STAGED_EPILOGUE_REDUCE = 3
} moe_forward_path;

/* device status bits */
#define MOE_DEV_TIMEOUT 1
#define MOE_DEV_BAD_EXPERT_MAP 2
#define MOE_DEV_BAD_INDEX 4      /* a row index outside the input or output; the row is skipped */

/* ------------------------------------------------------------------------------------------
 * Route preparation (lmdeploy PR #4857, section "Changes": sorted indices and compact blocks;
 * its review note asks that the local-expert slice and block_m be validated before launch).
 *
 * Routes are the M*k entries of topk_ids [M, k] (int32 global expert ids), numbered r = t*k + j.
 * A route is dropped when its id is < 0 or >= E, or when expert_map (int32 [E], nullable) sends
 * it to -1; expert_map maps a global id to a local expert in [0, E_local).  Without a map,
 * E_local must equal E.
 *
 * Outputs (device, int32):
 *   sorted_idx   [B_cap * block_m]  stable counting sort of the kept routes by local expert
 *                                   (experts ascending, route id ascending inside an expert);
 *                                   every expert's run is padded with -1 to a multiple of
 *                                   block_m; slots past the last block are -1.  Slot
 *                                   b*block_m + i is row i of block b.
 *   block_expert [B_cap]            local expert of block b, -1 for b >= num_blocks.  Only
 *                                   experts that received routes own blocks.
 *   num_blocks   [1]                number of blocks.
 *   expert_count [E_local]          kept routes per local expert.
 *   expert_offset[E_local + 1]      exclusive scan of the padded counts (slot of each run);
 *                                   nullable.
 *   route_slot   [M * k]            inverse of sorted_idx: the slot of route r, -1 when the
 *                                   route is dropped; nullable.
 * B_cap = moe_block_capacity(M, k, E_local, block_m) = ceil(M*k/block_m) + min(E_local, M*k).
 * k <= E (MOE_ERR_ARG otherwise).
 * block_m in {16, 32, 64, 128}.  path: AUTO takes one warp of one CTA for M*k <= 32 (a
 * match-any rank per route), the single-CTA sort when M*k <= 8192 and E_local <= 512
 * (measured faster than the multi-CTA launches there on GB300; the pages switch at 2048) and
 * the multi-CTA count/scan/scatter otherwise; the others force a path (SINGLE_CTA needs
 * M*k <= 8192 and E_local <= 2048).
 * workspace: moe_route_prepare_workspace_bytes(...) bytes, 256-byte aligned (only the multi-CTA
 * path uses it; the single-CTA path accepts a null workspace).  An expert_map entry outside [-1, E_local) drops that route and sets
 * MOE_DEV_BAD_EXPERT_MAP.
 * ------------------------------------------------------------------------------------------ */
MOEFP8_API int moe_block_capacity(int M, int k, int E_local, int block_m);
MOEFP8_API size_t moe_route_prepare_workspace_bytes(int M, int k, int E_local, int block_m);
MOEFP8_API int moe_route_prepare(const int32_t* topk_ids, int M, int k, int E, const int32_t* expert_map,
                      int E_local, int block_m, moe_route_path path, int32_t* sorted_idx,
                      int32_t* block_expert, int32_t* num_blocks, int32_t* expert_count,
                      int32_t* expert_offset, int32_t* route_slot, void* workspace,
                      size_t ws_bytes, cudaStream_t stream);

/* Allocation-free route preparation (no counterpart in the pages; added for callers that
 * cannot allocate).  Some callers have no way to obtain device memory for a workspace: a host
 * that owns every byte of device memory and gives this library neither an allocator nor a
 * workspace, or code that must not allocate at all because allocation would synchronise the
 * device or is forbidden where it runs.  This variant of the multi-CTA route preparation keeps
 * its scratch (per-chunk expert histograms, per-expert slot offsets, a ticket counter) in a
 * fixed array inside the library instead: 266,752 bytes of device memory on every GPU that
 * loads the library, held until the process exits.  It allocates nothing and calls no
 * allocating routine.
 *   Arguments and outputs are those of moe_route_prepare (always the multi-CTA path), without
 *   the workspace.  Limits: M*k <= 65536 routes and E_local <= 1024; larger sizes return
 *   MOE_ERR_ARG with nothing enqueued.
 *   Set-up: the first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress while that device is current; make that first call before any stream
 *   capture.
 *   Sharing: every call on a device uses the same array and leaves its contents behind (the
 *   ticket counter is cleared on the stream at the start of each call).  Calls whose execution
 *   overlaps on the GPU -- on different streams, or from different threads -- race on the array
 *   and give wrong results; serialise them. */
MOEFP8_API int moe_route_prepare_noalloc(const int32_t* topk_ids, int M, int k, int E,
                                         const int32_t* expert_map, int E_local, int block_m,
                                         int32_t* sorted_idx, int32_t* block_expert,
                                         int32_t* num_blocks, int32_t* expert_count,
                                         int32_t* expert_offset, int32_t* route_slot,
                                         cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Block-FP8 grouped GEMM over the active expert blocks (lmdeploy PR #4956, section
 * "Active-expert block scheduling"; lmdeploy PR #4857, transposed MMA for small block_m;
 * vLLM PR #53875, "FP8 W8A8 block shape [128, 128]").
 *
 * For every block b < num_blocks (expert e = block_expert[b]) and every slot s of b whose
 * route sorted_idx[s] >= 0:
 *   y[s, n] = sum_kb ( sum_{i in kb} a_q[s, i] * w_q[e, n, i] ) * a_s[s, kb] * w_s[e, n/128, kb]
 * accumulated in fp32.  Work is launched for real blocks only (num_blocks is read on the
 * device); pad slots are neither read for output nor written.
 * The activation rows are in SLOT order for both projections, not in token order: row s of
 * a_q is the input of the route in slot s.  The pages' kernels read token rows t = route / k
 * through the sorted indices inside the GEMM; here the gather happens before the GEMM (the
 * layer's input quantisation writes each token's codes to its routes' slots, e.g.
 * silu_mul_quant_fp8(IDENTITY, row_map = route_slot, row_div = k)), so that every GEMM operand
 * is a plain 2-D tensor tile.  A caller with token-ordered activations must gather them first.
 *   a_q  [a_rows, K] E4M3, rows in SLOT order (a_rows >= B_cap*block_m); a_s [a_rows, K/128] f32.
 *   w_q  [E_local, N_out, K] E4M3 (K contiguous) for MOE_WEIGHTS_ROW_MAJOR, or the tiled
 *        regrouping of it for MOE_WEIGHTS_TILED; w_s [E_local, N_out/128, K/128] f32.
 *   out  GATE_UP: row = slot s (out_rows >= B_cap*block_m);
 *        DOWN:    row = route sorted_idx[s] (out_rows > every route id, normally M*k).
 *   out_dtype BF16: out is [out_rows, N_out] bf16 (round to nearest even), splits must be 1.
 *   out_dtype F32 : out is [splits, out_rows, N_out] f32; split p holds the partial sum over
 *                   K-blocks [p*KB/splits, (p+1)*KB/splits) (KB = K/128), 1 <= splits <= KB.
 * K and N_out multiples of 128; block_m in {16, 32, 64, 128}; every pointer 16-byte aligned.
 * ------------------------------------------------------------------------------------------ */
MOEFP8_API int moe_blockfp8_grouped_gemm(moe_proj proj, const uint8_t* a_q, const float* a_s, int a_rows,
                              int K, const uint8_t* w_q, const float* w_s, int E_local, int N_out,
                              moe_weight_layout w_layout, const int32_t* sorted_idx,
                              const int32_t* block_expert,
                              const int32_t* num_blocks, int B_cap, int block_m, void* out,
                              moe_dtype out_dtype, int out_rows, int splits, cudaStream_t stream);

/* Weight regrouping for MOE_WEIGHTS_TILED (done once when the weights are loaded; not part of
 * the per-forward path): w_tiled[e][nt][kb][r][c] = w_q[e][nt*128 + r][kb*128 + c].  A tiled
 * weight tile is one contiguous 16 KB read for the GEMM's TMA instead of 128 rows of 128 bytes
 * that lie K bytes apart.  N_out and K multiples of 128; both pointers 16-byte aligned; the
 * buffers must not overlap. */
MOEFP8_API int moe_blockfp8_pack_weights(const uint8_t* w_q, int E_local, int N_out, int K,
                                         uint8_t* w_tiled, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Fused (optionally clamped) SiLU-and-mul with per-128-group dynamic E4M3 quantisation
 * (vLLM PR #53875, section "Purpose"; lmdeploy PR #4956, "Fused SwiGLU and FP8 quantization").
 *
 * Per work row i and group g of 128 columns: the activation a (see moe_act) is materialised in
 * BF16 in registers only; s = max(amax|a|, 1e-10) / 448 (IEEE fp32 division), rounded up to a
 * power of two for MOE_SCALE_UE8M0; q = e4m3_rn_satfinite(a / s) (IEEE division).
 *   in  BF16 [in_rows, W] (in_dtype BF16, in_splits 1) or F32 [in_splits, in_rows, W]
 *       (in_dtype F32: split partial sums, added in split order in fp32 and rounded to BF16
 *       first); W = N for IDENTITY, 2N otherwise.
 *   out_q [out_rows, N] E4M3; out_s [out_rows, N/128] f32.
 * Rows: work row i in [0, rows) reads input row i and writes output row i, unless row_map
 *   (nullable int32 [rows]) is given: then m = row_map[i] < 0 skips the row, the output row is
 *   m and the input row is i / row_div (row_div >= 1) or m (row_div == 0).  This is how the
 *   layer gathers token rows into expert-sorted slot order (row_map = route_slot, row_div = k).
 * Expert filter (nullable row_expert [rows] int32 global ids): a work row whose id is < 0,
 *   >= E, or sent to -1 by expert_map (nullable, [E]) is skipped.
 * Skipped rows leave out_q / out_s as they were.  An input or output row index past in_rows or
 * out_rows skips the row and sets MOE_DEV_BAD_INDEX.  clamp_limit: +inf for none.
 * strategy: PER_GROUP launches one warp per pair of quant groups with no loop (launch-bound
 * decode without a filter), PERSISTENT a grid-stride kernel of as many CTAs as are resident at
 * once; AUTO picks
 * PER_GROUP when there is no filter or map and rows*N < 2^20.
 * N multiple of 128; rows * N/128 < 2^31; in and out_q 16-byte aligned.
 * ------------------------------------------------------------------------------------------ */
MOEFP8_API int silu_mul_quant_fp8(moe_act act, const void* in, moe_dtype in_dtype, int in_splits,
                       int in_rows, int rows, int N, float clamp_limit, moe_scale_fmt fmt,
                       const int32_t* row_expert, const int32_t* expert_map, int E,
                       const int32_t* row_map, int row_div, int out_rows, uint8_t* out_q,
                       float* out_s, moe_quant_strategy strategy, cudaStream_t stream);

/* The unfused first half of the two-kernel path (lmdeploy PR #4956, "Motivation"): writes the
 * BF16 SiLU*mul result out [rows, N] from in [rows, 2N].  act must not be IDENTITY.  Used as
 * the separate-kernel arm that the fused kernel is compared with.  The expert filter
 * (row_expert nullable [rows] global ids, expert_map nullable [E]) skips the same rows as in
 * silu_mul_quant_fp8 and leaves their output rows untouched (vLLM PR #53875, "Kernel
 * microbenchmarks": the filter applies in both arms). */
MOEFP8_API int silu_and_mul_bf16(moe_act act, const void* in, int rows, int N, float clamp_limit,
                                 const int32_t* row_expert, const int32_t* expert_map, int E,
                                 void* out, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * moe_reduce (lmdeploy PR #4228 "Moe Reduce kernel"): weighted top-k sum back to one row per
 * token, out[t, h] = bf16( sum_j w[t, j] * z[t*k + j, h] ) over the kept routes in j order,
 * fp32 accumulation with one fused multiply-add per term.  Dropped routes contribute nothing
 * and their z rows are never read.  A route is dropped by the same rule as in route
 * preparation: id < 0, id >= E, or an expert_map entry outside [0, E_local) (-1, or an invalid
 * entry for which route preparation gave the route no slot).
 *   z [M*k, H] bf16 (route order); topk_w [M, k] f32; topk_ids [M, k] int32;
 *   expert_map nullable [E] (without it E_local must equal E); out [M, H] bf16.  H multiple
 *   of 8, k <= 32, M * ceil(H/256) < 2^31; pointers 16-byte aligned.
 * ------------------------------------------------------------------------------------------ */
MOEFP8_API int moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
               const int32_t* expert_map, int M, int k, int E, int E_local, int H, void* out,
               cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * The whole layer (lmdeploy PR #4956, sections "Active-expert block scheduling" and "Fused SwiGLU
 * and FP8 quantization"; lmdeploy PR #4228 for the final weighted sum): route preparation ->
 * input quantisation (gathered into slot order) -> gate/up grouped GEMM -> fused SiLU*mul +
 * quantisation -> down grouped GEMM -> moe_reduce.
 *   x [M, H] bf16 (16-byte aligned); topk_ids / topk_w [M, k]; expert_map nullable [E]
 *   (E_local local experts); wgu_q [E_local, 2N, H] E4M3 + wgu_s [E_local, 2N/128, H/128] f32
 *   (gate rows 0..N-1, up rows N..2N-1); wd_q [E_local, H, N] E4M3 + wd_s [E_local, H/128,
 *   N/128] f32; both weight tensors in w_layout (row-major, or tiled by
 *   moe_blockfp8_pack_weights); act SILU_MUL or SILU_MUL_GATE_UPPER; clamp_limit (+inf = none);
 *   act_fmt for the dynamic activation scales (input and intermediate); block_m 0 = chosen from
 *   the shape.  out [M, H] bf16.  workspace: moe_blockfp8_workspace_bytes(...) bytes, 256-byte
 *   aligned (the same size serves both paths).
 * path FUSED: after route preparation ONE persistent kernel with one CTA per SM runs the rest;
 *   its phases are separated by counters in the workspace, so the kernel needs all its CTAs
 *   resident at once: do not run it concurrently with other work that occupies SMs for its
 *   whole duration (every wait is bounded; such a run ends with MOE_DEV_TIMEOUT in the device
 *   status word instead of hanging).  The gate/up K range is dealt to the SMs in equal pieces,
 *   so the fp32 summation order of the gate/up partial sums (not the arithmetic of any stage)
 *   depends on the SM count.  path STAGED: one launch per stage.  path STAGED_EPILOGUE_REDUCE:
 *   the down GEMM also does the weighted top-k sum (lmdeploy PR #4228's reduce, with per-token
 *   ownership): once a unit has stored its z rows, each row counts itself in a counter of its
 *   (token, 128-column tile); the arrival that completes a token's kept routes sums that
 *   token's 128 columns in top-k order with the same fp32 fused multiply-adds as moe_reduce,
 *   so the output is bitwise the STAGED output.  AUTO: see moe_forward_path_for.
 * H and N multiples of 128; k <= E.  The staged path's reduce takes k <= 32: STAGED with a
 * larger k is refused (MOE_ERR_ARG, nothing enqueued) and AUTO then takes FUSED, which has no
 * top-k limit.  All stages run on `stream` with no host synchronisation, so the call can be
 * captured in a CUDA graph.
 * x, topk_ids, topk_w and out may be device memory or pinned host memory that the device sees
 * at the same address (cudaHostAlloc / cudaHostRegister under unified addressing; check with
 * moe_pointer_device_accessible): the input quantisation, route preparation and reduce kernels
 * read x, topk_ids and topk_w and write out directly there (each byte crosses the host link
 * once; the call is still asynchronous, so the host reads out after synchronising `stream`).
 * The weights, expert_map and workspace must be device memory.
 * ------------------------------------------------------------------------------------------ */
MOEFP8_API size_t moe_blockfp8_workspace_bytes(int M, int k, int E, int E_local, int H, int N, int block_m);
MOEFP8_API int moe_blockfp8_forward(const void* x, const int32_t* topk_ids, const float* topk_w, int M,
                         int k, int E, const int32_t* expert_map, int E_local, int H, int N,
                         const uint8_t* wgu_q, const float* wgu_s, const uint8_t* wd_q,
                         const float* wd_s, moe_weight_layout w_layout, moe_act act,
                         float clamp_limit, moe_scale_fmt act_fmt, int block_m,
                         moe_forward_path path, void* out, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);
/* Where the forward keeps its intermediate tensors inside the workspace: offsets[i] is the
 * byte offset of region i (moe_ws_region) for these sizes and block_m (0 = the forward's own
 * choice).  For inspecting a finished forward (the tests compare these tensors with the
 * oracle); the regions are rewritten by every forward.  Host only.  Regions and layouts
 * (slots = B_cap * block_m, KB = H/128, GN = N/128, S = the gate/up split count of
 * moe_blockfp8_plan):
 *   SORTED_IDX int32 [slots], BLOCK_EXPERT int32 [B_cap], NUM_BLOCKS int32 [1],
 *   EXPERT_COUNT int32 [E_local], EXPERT_OFFSET int32 [E_local + 1], ROUTE_SLOT int32 [M*k]:
 *     the outputs of moe_route_prepare;
 *   XQ  E4M3 [slots, H]: the quantised input, row = slot of a kept route;
 *   XS  f32 scales of XQ: STAGED [slots, KB]; FUSED K-block major [KB, slots];
 *   GU  gate/up partial sums: STAGED f32 [S, slots, 2N] (split p covers K-blocks
 *       [p*KB/S, (p+1)*KB/S)), or with S = 1 the sum rounded to BF16, bf16 [slots, 2N];
 *       FUSED f32 [pieces, num_blocks * block_m, 2N], piece q of a
 *       128-column tile is its q-th stream-K range (see moe_blockfp8_forward);
 *   AQ  E4M3 [slots, N]: the quantised SiLU*mul activation; AS its scales: STAGED
 *       [slots, GN]; FUSED [GN, slots];
 *   Z   bf16 [M*k, H]: the down projection's output, route order.
 * Returns MOE_OK or MOE_ERR_ARG. */
typedef enum {
    MOE_WS_SORTED_IDX = 0, MOE_WS_BLOCK_EXPERT = 1, MOE_WS_NUM_BLOCKS = 2, MOE_WS_EXPERT_COUNT = 3,
    MOE_WS_EXPERT_OFFSET = 4, MOE_WS_ROUTE_SLOT = 5, MOE_WS_XQ = 6, MOE_WS_XS = 7, MOE_WS_GU = 8,
    MOE_WS_AQ = 9, MOE_WS_AS = 10, MOE_WS_Z = 11, MOE_WS_REGIONS = 12
} moe_ws_region;
MOEFP8_API int moe_blockfp8_workspace_layout(int M, int k, int E, int E_local, int H, int N,
                                             int block_m, size_t* offsets /*[MOE_WS_REGIONS]*/);

/* The path moe_blockfp8_forward takes for path = AUTO at these sizes (FUSED or STAGED). */
MOEFP8_API int moe_forward_path_for(int M, int k, int E, int E_local, int H, int N);

/* block_m the forward uses when called with block_m = 0: 16 up to M = 256 tokens, 32 above
 * (measured fastest on GB300 for the decode, expert-parallel and prefill shapes). */
MOEFP8_API int moe_forward_block_m(int M, int k, int E_local, int H, int N);

/* The launch plan moe_blockfp8_forward uses for these sizes: block_m, B_cap (blocks of
 * capacity) and the split-K count of the gate/up GEMM (its fp32 partials are summed by the
 * fused activation kernel).  Host only; returns MOE_OK or MOE_ERR_ARG. */
MOEFP8_API int moe_blockfp8_plan(int M, int k, int E, int E_local, int H, int N, int block_m,
                                 int* out_block_m, int* out_B_cap, int* out_splits);

/* Whether the staged forward's gate/up and down GEMMs (*gate_up, *down: 1 or 0) hand out the
 * last quarter of their work units from a counter in the workspace instead of splitting all of
 * them statically over the SMs: only when a GEMM's expected active-expert weight stream is long
 * (at least 8 MB per SM, 2.5 MiB per SM at block_m 16), where the SMs' differing streaming
 * rates would otherwise leave a tail.  A scheduling choice of this library, no counterpart in
 * the pages; every unit is computed exactly as in the static split, so the results are the
 * same bit for bit.  Host only; MOE_OK, or MOE_ERR_ARG for bad sizes or null outputs. */
MOEFP8_API int moe_blockfp8_dynamic_tail(int M, int k, int E, int E_local, int H, int N,
                                         int block_m, int* gate_up, int* down);

/* The plan of moe_blockfp8_plan and moe_blockfp8_dynamic_tail for a device with `sms` SMs
 * instead of the current device (152 on a GB300): block_m, block capacity, gate/up split
 * count and the two dynamic-tail flags (1 or 0).  Any output pointer may be null.  It lets a
 * host without that device compute the plan, and tests check the plan's rules without a GPU.
 * A scheduling choice of this library, no counterpart in the pages.  Host only; MOE_OK, or
 * MOE_ERR_ARG for bad sizes or sms <= 0. */
MOEFP8_API int moe_blockfp8_plan_for_sms(int M, int k, int E, int E_local, int H, int N,
                                         int block_m, int sms, int* out_block_m, int* out_B_cap,
                                         int* out_splits, int* out_dyn_gate_up,
                                         int* out_dyn_down);

/* ------------------------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------------------------ */
/* Text of the last error on this thread ("" if none).  The pointer stays valid until the next
 * call on this thread. */
MOEFP8_API const char* moe_last_error_string(void);
/* Reads (synchronously) the status word of the current device into *status; reset != 0 clears
 * it afterwards.  Returns MOE_OK or MOE_ERR_LAUNCH. */
MOEFP8_API int moe_get_device_status(int* status, int reset);
/* 1 if the current device is an sm_103 GPU the library was built for, else 0. */
MOEFP8_API int moe_device_supported(void);
/* Test hook for the bounded waits (no counterpart in the pages).  The next path-FUSED forward
 * launched from the calling thread treats block `block` of the layer as one gate/up piece
 * short, so the activation step's wait for that block can never complete, and uses
 * wait_limit_ns (at most the default 2 s) as the limit of its counter waits.  Every index and
 * address stays valid: the wait runs out, MOE_DEV_TIMEOUT is set in the device status word,
 * the kernel drains its copies and tensor-core work, frees its tensor memory and returns, and
 * the output of that call is undefined.  The setting applies to one launch and is then
 * cleared.  Returns MOE_OK, or MOE_ERR_ARG for block < 0 or a limit outside (0, 2 s]. */
MOEFP8_API int moe_debug_inject_stall(int block, unsigned long long wait_limit_ns);

/* The binary architecture version of the library's kernels as the CUDA runtime reports it for
 * the current device (cudaFuncGetAttributes binaryVersion, 103 for sm_103a code), or -1 when
 * it cannot be queried (no device). */
MOEFP8_API int moe_kernel_binary_version(void);
/* 1 if kernels on the current device can dereference p as it is: device memory of this device,
 * managed memory, or pinned host memory mapped at the same address; else 0 (also for null and
 * for pageable host memory).  Host only, no device work. */
MOEFP8_API int moe_pointer_device_accessible(const void* p);

#ifdef __cplusplus
}
#endif
#endif /* MOEFP8_H */
