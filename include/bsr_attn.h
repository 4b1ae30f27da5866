/*
 * bsr_attn.h -- C ABI of the GB300 (sm_103a) block-sparse attention library.
 *
 * Block-sparse attention computes softmax(scale * Q K^T) V over the stored
 * 128 x 128 blocks of a block mask given in BSR form (block-row pointers and
 * block-column indices); every score outside a stored block is removed.  The
 * forward pass also returns the fp32 row statistics, and the backward pass
 * computes dQ by walking block rows and dK / dV by walking block columns of
 * a BSC transpose built on the host, so that every output tile has exactly
 * one writer and no atomics are used.
 *
 * Sources: "trnsparse 0.7.0 -> 0.9.0" diff (CHANGELOG [0.8.0], native path:
 * static-structure kernels, attn_fwd_static / attn_bwd_static; CHANGELOG
 * [0.9.0], one writer per output tile, bf16 operands with fp32 accumulation
 * and fp32 statistics) and "trnsparse 0.4.1 -> 0.6.0" diff (CHANGELOG
 * [0.5.0] delta identity; [0.5.1] dQ row-first and dK/dV column-first
 * kernels, host-built BSC view, returned row_max / row_denom; [0.6.0]
 * head_dim 256 and 512 by 128-wide chunks of the QK^T contraction).
 *
 * Conventions shared by every entry point:
 *  - Dense tensors are [batch, heads, seq, head_dim], contiguous, row-major,
 *    described by a bsr_tensor whose `data` is a DEVICE pointer, 16-byte
 *    aligned (inputs are read by TMA, outputs written with 16- and 32-byte
 *    vector stores; a misaligned pointer is BSR_ERR_INVALID_ARG).  All dense
 *    tensors of one call have the same shape and dtype.  Supported:
 *    head_dim in {64, 128, 256, 512}; dtype BSR_F32, BSR_BF16 or BSR_F16
 *    (16-bit operands are multiplied on the tensor cores with fp32
 *    accumulation, and outputs are rounded to the operand type; the
 *    statistics are fp32 for every dtype, as the "trnsparse 0.7.0 -> 0.9.0"
 *    diff, CHANGELOG [0.9.0], has them for fp16 and bf16 inputs);
 *    seq = n_brows * 128; batch, heads >= 1.
 *  - Statistics row_max / row_denom are fp32 DEVICE arrays [batch, heads, seq].
 *    row_max is the maximum of the scaled scores scale * q.k of the row over
 *    its stored blocks (natural-log units) and row_denom the sum of
 *    exp(scale * q.k - row_max) over the same scores.  A block row with no
 *    stored block gets O = 0, row_max = -inf, row_denom = 0.
 *  - The mask is shared by every (batch, head).  row_ptr / col_idx /
 *    col_ptr / row_idx passed to the kernels are int32 DEVICE arrays; columns
 *    ascend without repeats inside a row (bsr_validate checks this on host).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous on it.  The caller owns every buffer; the library allocates
 *    only stream-ordered scratch (cudaMallocAsync / cudaFreeAsync on `stream`).
 *    The attention calls can be recorded by stream capture into a CUDA graph
 *    and replayed (their second stream joins the capture through events);
 *    make the first call of a process outside capture, since it sets kernel
 *    attributes and creates that stream.
 *  - Every function returns a bsr_status; nothing throws across the ABI and
 *    there is no fallback path.  bsr_last_error() gives a message for the
 *    last failure on the calling thread.
 */
#ifndef BSR_ATTN_H
#define BSR_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { BSR_F32 = 0, BSR_BF16 = 1, BSR_F16 = 2 } bsr_dtype;

typedef enum {
  BSR_OK = 0,
  BSR_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad structure */
  BSR_ERR_UNSUPPORTED = 2,   /* head_dim / dtype / block outside the supported set */
  BSR_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  BSR_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up (reported by bsr_attn_check) */
  BSR_ERR_DEVICE_CHECK = 5   /* a device-side bounds check failed (reported by bsr_attn_check) */
} bsr_status;

typedef struct {
  void* data;        /* device pointer (16-byte aligned) to [batch, heads, seq, head_dim] elements */
  int32_t dtype;     /* bsr_dtype */
  int32_t batch;
  int32_t heads;
  int32_t seq;
  int32_t head_dim;
} bsr_tensor;

/*
 * Forward pass ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0]:
 * attn_fwd_static, one launch with the softmax statistics kept on chip, no
 * K/V gather and no per-block score round trip through HBM).
 *
 *   O[i]         = sum_j P[i,j] V[j],   P = softmax over stored j of scale * Q[i].K[j]
 *   row_max[i]   = max over stored j of scale * Q[i].K[j]
 *   row_denom[i] = sum over stored j of exp(scale * Q[i].K[j] - row_max[i])
 *
 * Q, K, V, O: dense tensors (device), O written in the operands' dtype.
 * row_ptr: int32 [n_brows + 1] (device); col_idx: int32 [row_ptr[n_brows]] (device).
 * block must be 128.  scale is usually 1/sqrt(head_dim).
 * Errors: BSR_ERR_INVALID_ARG for null pointers or mismatched shapes,
 * BSR_ERR_UNSUPPORTED for block != 128, head_dim or dtype outside the set,
 * BSR_ERR_CUDA when a launch fails.  Nothing is written on error.
 */
bsr_status bsr_attn_fwd(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                        const int32_t* row_ptr, const int32_t* col_idx, int32_t n_brows,
                        int32_t block, float scale,
                        bsr_tensor* O, float* row_max, float* row_denom, void* stream);

/*
 * The statistics-first variant of the forward pass ("trnsparse 0.4.1 ->
 * 0.6.0" diff, CHANGELOG [0.4.3]: first the row statistics over the row's
 * stored blocks, then the output with P = exp(scale * Q[i].K[j] - row_max[i])
 * / row_denom[i]), for comparison with bsr_attn_fwd: same arguments, same
 * results up to rounding, two tensor-core launches (the first reads Q and K
 * only and writes row_max / row_denom, the second reads them back).
 * Supported for BSR_BF16 / BSR_F16 operands with head_dim 64 or 128;
 * otherwise BSR_ERR_UNSUPPORTED.  Other errors as bsr_attn_fwd.
 */
bsr_status bsr_attn_fwd_two_pass(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                                 const int32_t* row_ptr, const int32_t* col_idx, int32_t n_brows,
                                 int32_t block, float scale,
                                 bsr_tensor* O, float* row_max, float* row_denom, void* stream);

/*
 * Block-sparse times dense ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG
 * [0.8.0]: bsr_spmm_static walks exactly the stored blocks and addresses X
 * by block column; [0.9.0]: bf16 operands with fp32 accumulation):
 *
 *   Y[m*128 + i, c] = sum over stored blocks j of block row m, k = col_idx[j],
 *                     sum_t blocks[j][i][t] * X[k*128 + t, c]
 *
 * blocks: [nnzb][128][128] row-major (device), the stored blocks in BSR order;
 * row_ptr: int32 [n_brows + 1], col_idx: int32 [nnzb] (device), columns in
 * [0, n_bcols); X: [n_bcols * 128][n_cols], Y: [n_brows * 128][n_cols],
 * row-major (device); blocks, X and Y have element type `dtype` (BSR_BF16 or
 * BSR_F16; products accumulated in fp32, Y rounded to the element type).
 * Pointers 16-byte aligned; block must be 128; n_cols a positive multiple
 * of 64.  A block row with no stored block gets Y rows of zeros.
 * Errors: BSR_ERR_INVALID_ARG (null / misaligned pointer, bad size),
 * BSR_ERR_UNSUPPORTED (block, dtype, n_cols), BSR_ERR_CUDA; a col_idx
 * outside [0, n_bcols) or a row_ptr outside [0, nnzb] is skipped on the
 * device and reported by bsr_attn_check as BSR_ERR_DEVICE_CHECK.
 */
bsr_status bsr_spmm(const void* blocks, int32_t dtype, const int32_t* row_ptr, const int32_t* col_idx,
                    int32_t n_brows, int32_t n_bcols, int32_t nnzb, int32_t block, const void* X,
                    int32_t n_cols, void* Y, void* stream);

/*
 * Fused screened SpMM ("trnsparse 0.7.0 -> 0.9.0" diff, docs:
 * screened_spmm(A, diag, B, threshold) fuses the Schwarz pair bound, the
 * threshold mask and the matmul into one dispatch):
 *
 *   C = (A o M) B,  M[i, j] = sqrt(|diag[i]|) * sqrt(|diag[j]|) > sqrt(threshold)
 *
 * with the square roots, the product and the comparison in fp32.  A:
 * [n][n], B and C: [n][n_cols], row-major, element type `dtype` (BSR_BF16
 * or BSR_F16; fp32 accumulation, C rounded to the element type); diag: fp32
 * [n]; all device pointers, 16-byte aligned.  n a multiple of 128 up to
 * 65536, n_cols a positive multiple of 64, threshold finite and >= 0.
 * 128 x 128 tiles of A whose pairs all fail the bound are never read.
 * Errors: BSR_ERR_INVALID_ARG (null / misaligned pointer, bad size or
 * threshold), BSR_ERR_UNSUPPORTED (dtype, n, n_cols), BSR_ERR_CUDA.
 */
bsr_status bsr_screened_spmm(const void* A, const float* diag, const void* B, int32_t dtype, int32_t n,
                             int32_t n_cols, float threshold, void* C, void* stream);

/*
 * Backward pass ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.5.0] delta
 * identity D_i = dO_i . O_i; [0.5.1] _attn_bwd_dq_kernel row-first and
 * _attn_bwd_dkdv_kernel column-first over the host-built BSC view, no
 * atomic scatter; "trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0]
 * attn_bwd_static).
 *
 *   P = exp(scale * Q K^T - row_max) / row_denom on stored blocks,
 *   dV = P^T dO;  dS = P * (dO V^T - D);  dQ = scale dS K;  dK = scale dS^T Q.
 *
 * Q, K, V, O, dO: dense inputs (device); O, row_max, row_denom from
 * bsr_attn_fwd with the same scale.  row_ptr / col_idx: the BSR lists;
 * col_ptr: int32 [n_bcols + 1] and row_idx: int32 [nnzb], the BSC transpose
 * from bsr_build_bsc (rows ascending inside a column); all device arrays.
 * `scale` must equal the forward's (the signature carries it explicitly).
 * dQ, dK, dV: dense outputs (device), every element written (tiles of empty
 * block columns / rows are written as zeros).
 * Scratch: two fp32 [batch, heads, seq] arrays (delta, base-2 log-sum-exp),
 * stream-ordered.
 * Errors as for bsr_attn_fwd.
 */
bsr_status bsr_attn_bwd(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                        const bsr_tensor* O, const bsr_tensor* dO,
                        const float* row_max, const float* row_denom,
                        const int32_t* row_ptr, const int32_t* col_idx,
                        const int32_t* col_ptr, const int32_t* row_idx,
                        float scale,
                        bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV, void* stream);

/*
 * Backward pass that allocates nothing.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory, either
 * because another allocator already owns the device's memory (a framework's
 * caching allocator, a serving runtime's pools) or because their hot path
 * must not call into the CUDA allocator.  Same arguments, results and errors
 * as bsr_attn_bwd, but its scratch (delta and log-sum-exp per row, and the
 * two work lists) comes from a fixed array in the library's static device
 * memory (9 MiB per GPU that loads the library, held until the process
 * exits) instead of cudaMallocAsync.  Long block rows / columns are not
 * split into chunks on this path (that would need partial-result buffers).
 * Limits: batch * heads * seq <= 1,048,576; for fp32 operands, whose bf16
 * pieces (24 bytes per element of Q) share the array, also batch * heads *
 * seq * head_dim up to about 390,000; beyond that BSR_ERR_INVALID_ARG.
 * All calls share the array: calls whose kernels overlap on the GPU race, so
 * order them on one stream.  The first call on a device (with that device
 * current) looks up the array's device address; make it before any stream
 * capture.  That address is kept for the rest of the process, so this entry
 * point must not be called after cudaDeviceReset has destroyed the device's
 * primary context (the array would move, the kept address would not).
 */
bsr_status bsr_attn_bwd_noalloc(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                                const bsr_tensor* O, const bsr_tensor* dO,
                                const float* row_max, const float* row_denom,
                                const int32_t* row_ptr, const int32_t* col_idx,
                                const int32_t* col_ptr, const int32_t* row_idx,
                                float scale,
                                bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV, void* stream);

/*
 * Reusable plans.  A plan holds, for one block mask and one operand shape,
 * the work lists of the forward / dQ walk and of the dK / dV walk, built
 * once, plus every scratch array the passes need (split-row partial
 * results, the fp32 operands' bf16 pieces, delta and lse2): a call on a plan
 * launches only the attention kernels and the backward's delta pass, with
 * no planner and no allocation.  This follows the pages' static-structure
 * design ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0]: kernels built
 * once per structure and reused) with the structure kept as data.
 *
 * bsr_plan_create: row_ptr [n_brows+1], col_idx [nnzb], col_ptr [n_brows+1]
 *   and row_idx [nnzb] are int32 DEVICE arrays (the BSR lists and their BSC
 *   transpose from bsr_build_bsc; the grid is square, n_bcols = n_brows);
 *   the plan copies them, so the caller may free or change them afterwards.
 *   batch, heads, head_dim and dtype fix the operand shape [batch, heads,
 *   n_brows * 128, head_dim] the plan serves.  The call reads nnzb from the
 *   device (it synchronises `stream`), allocates the plan's device memory
 *   with cudaMalloc on the current device and builds the lists on `stream`;
 *   use the plan on that stream (or synchronise first).  *out receives the
 *   handle (NULL on failure).  The plan also holds a dS workspace of
 *   batch * heads * nnzb tiles of 32 KiB (64 KiB for fp32 operands: dS in
 *   two bf16 pieces): the dK/dV (or dK) walk stores each dS tile there and
 *   the plan's dQ walk sums dS K over them instead of recomputing the
 *   scores (head_dim 256 / 512 and fp32 operands: as many P^T tiles again,
 *   which the dV walk sums P^T dO over).  It reads col_idx and row_idx to the host to map every BSC entry
 *   to its BSR position, and if that workspace cannot be allocated the
 *   plan's dQ walk recomputes the scores instead (same results within the
 *   tolerances).  Errors:
 *   BSR_ERR_INVALID_ARG for null pointers, bad sizes, row_ptr / col_ptr whose
 *   last entries disagree, or a BSC entry that is not a stored block of the
 *   BSR lists; BSR_ERR_UNSUPPORTED for a head_dim / dtype outside the
 *   supported set; BSR_ERR_CUDA when an allocation or copy fails.
 * bsr_plan_destroy: frees the plan (cudaFree: synchronises the device).
 *   NULL is accepted.
 * bsr_attn_fwd_plan / bsr_attn_bwd_plan: the same computations and the same
 *   argument meaning as bsr_attn_fwd / bsr_attn_bwd, with the structure taken
 *   from the plan.  The operands must have the plan's shape and dtype and the
 *   current device must be the plan's (BSR_ERR_INVALID_ARG otherwise).
 *   Calls on one plan share its scratch: order them on one stream (calls on
 *   different plans are independent).  After BSR_ERR_TIMEOUT from
 *   bsr_attn_check the plan's work counters may be left mid-launch: destroy
 *   the plan and build it again.
 */
typedef struct bsr_plan_s bsr_plan;

bsr_status bsr_plan_create(const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
                           const int32_t* row_idx, int32_t n_brows, int32_t batch, int32_t heads,
                           int32_t head_dim, int32_t dtype, void* stream, bsr_plan** out);
bsr_status bsr_plan_destroy(bsr_plan* plan);
bsr_status bsr_attn_fwd_plan(const bsr_plan* plan, const bsr_tensor* Q, const bsr_tensor* K,
                             const bsr_tensor* V, float scale, bsr_tensor* O, float* row_max,
                             float* row_denom, void* stream);
bsr_status bsr_attn_bwd_plan(const bsr_plan* plan, const bsr_tensor* Q, const bsr_tensor* K,
                             const bsr_tensor* V, const bsr_tensor* O, const bsr_tensor* dO,
                             const float* row_max, const float* row_denom, float scale,
                             bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV, void* stream);

/*
 * bsr_plan_work_list: copies one of a plan's work lists to the host
 * (synchronises `stream`), for inspecting the schedule the persistent kernels
 * follow.  list 0: block rows (forward, dQ); 1: block columns (dK / dV);
 * 2: the second block-column list (the dK walk of the head_dim-256 / 512 and
 * fp32 kernels).  The items come in the order the kernels draw them: by
 * block count, longest first, and inside one count by line, ascending.  A
 * line longer than the per-CTA share Lmax = max(8, ceil(nnzb * H' / G)) is
 * cut into ceil(len / Lmax) chunks whose lengths differ by at most one,
 * longer chunks first ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.9.0]:
 * work balanced by stored blocks, one writer per output tile); lines with
 * no stored block get no item.  Item i goes to items[4 i .. 4 i + 3] as
 * (line, first, n, slot): the block row / column, the offset of its first
 * block in col_idx / row_idx, its block count, and -1 for a whole line or
 * the partial-result slot of a chunk (the chunks of one line have
 * consecutive slots).  items holds `cap` items (host memory, owned by the
 * caller).  info (host, 4 int32) receives the item count, G (the persistent
 * CTAs the plan serves), H' (the heads the planner counts: batch * heads,
 * times the output slices of the head_dim-256 / 512 and fp32 kernels) and
 * the number of distinct item lengths.  Errors: BSR_ERR_INVALID_ARG for a
 * null argument, a list outside 0..2 or too small a `cap`; BSR_ERR_CUDA
 * when a copy fails.
 */
bsr_status bsr_plan_work_list(const bsr_plan* plan, int32_t list, int32_t* items, int32_t cap, int32_t* info,
                              void* stream);

/*
 * Host helper: BSC transpose of a BSR block structure ("trnsparse 0.4.1 ->
 * 0.6.0" diff, CHANGELOG [0.5.1], _attn_bwd_gather, host-side BSC
 * construction).  All pointers are HOST arrays owned by the caller:
 * row_ptr_h [n_brows+1], col_idx_h [nnzb] in; col_ptr_h [n_bcols+1],
 * row_idx_h [nnzb] out.  Block rows ascend inside each block column.
 * Returns BSR_ERR_INVALID_ARG (and writes nothing) when the BSR lists fail
 * bsr_validate.
 */
bsr_status bsr_build_bsc(const int32_t* row_ptr_h, const int32_t* col_idx_h,
                         int32_t n_brows, int32_t n_bcols,
                         int32_t* col_ptr_h, int32_t* row_idx_h);

/*
 * Host helper: checks BSR lists (HOST arrays): row_ptr[0] = 0, row_ptr
 * non-decreasing, every col_idx in [0, n_bcols), strictly ascending inside a
 * row (no duplicates).  Returns BSR_OK or BSR_ERR_INVALID_ARG with a message.
 */
bsr_status bsr_validate(const int32_t* row_ptr_h, const int32_t* col_idx_h,
                        int32_t n_brows, int32_t n_bcols);

/*
 * Synchronises `stream`, then reads and clears the device status word that
 * the kernels set when a bounded wait gives up (BSR_ERR_TIMEOUT) or a device
 * bounds check fails (BSR_ERR_DEVICE_CHECK).  BSR_OK when neither happened.
 */
bsr_status bsr_attn_check(void* stream);

/*
 * Limit of the kernels' bounded device-side waits on the current device, in
 * nanoseconds (0 restores the default of 2 s).  No passage of the pages
 * defines it: every wait inside the kernels (pipeline barriers between the
 * copy, MMA and elementwise roles) gives up after this much wall time, the
 * kernel then drains its copies and MMAs, frees its tensor memory, returns,
 * and bsr_attn_check reports BSR_ERR_TIMEOUT.  Lowering the limit to a few
 * hundred nanoseconds makes those waits expire on purpose, which is how the
 * give-up path is tested; results of calls made under such a limit are
 * undefined.  The call synchronises the device before and after it changes
 * the limit; make it while no call of this library is in flight.
 */
bsr_status bsr_set_wait_limit(uint64_t ns);

/* Message for the last non-OK status returned on the calling thread. */
const char* bsr_last_error(void);

/*
 * Kernel timing for benchmarks.  While enabled, every kernel the library
 * launches is bracketed by CUDA events recorded on its launching stream.
 * bsr_profile_collect synchronises those events and returns, per kernel name,
 * the number of launches and their summed duration in ms since the last
 * collect, then clears the record.  Returns the number of entries written.
 */
typedef struct {
  char name[48];
  int32_t launches;
  float total_ms;
} bsr_kernel_time;

void bsr_profile_enable(int32_t on);
int32_t bsr_profile_collect(bsr_kernel_time* out, int32_t max_entries);

#ifdef __cplusplus
}
#endif

#endif /* BSR_ATTN_H */
