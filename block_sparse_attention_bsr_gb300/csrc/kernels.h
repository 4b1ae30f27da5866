// Kernel-side declarations: argument blocks and launchers for the attention
// kernels.  Shared by the C-ABI front end and the kernel translation units.
#pragma once

#include <mutex>

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace bsr {

// Device status word values (mirrors bsr_status).
enum : int { kStatusOk = 0, kStatusTimeout = BSR_ERR_TIMEOUT, kStatusDeviceCheck = BSR_ERR_DEVICE_CHECK };

struct Dims {
  int BH;      // batch * heads
  int S;       // sequence length (rows per head)
  int D;       // head_dim
  int nb;      // S / 128 block rows (= block columns)
  int dtype;   // bsr_dtype
  float scale;
};

struct FwdArgs {
  Dims d;
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* row_max;
  float* row_denom;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int32_t* plan;          // block-row plan (plan.cu)
  int G;                  // persistent CTAs the plan was built for
  float* part;            // partial results of split rows: O (128 x D) and 3 x 128 stats per tile
  void* pieces;           // fp32 operands: the three bf16 pieces of Q, K, V (wide_piece_bytes(d, 3))
  int* status;
};

struct BwdArgs {
  Dims d;
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const void* dO;
  const float* row_max;
  const float* row_denom;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const int32_t* col_ptr;
  const int32_t* row_idx;
  void* dQ;
  void* dK;
  void* dV;
  float* delta;  // [BH * S] scratch: D_i = dO_i . O_i
  float* lse2;   // [BH * S] scratch: row_max * log2(e) + log2(row_denom)
  int32_t* row_plan;   // block-row plan (dQ walk)
  int32_t* col_plan;   // block-column plan (dK/dV walk; the dV walk of the wide kernels)
  int32_t* col_plan2;  // block-column plan of the wide kernels' dK walk
  void* pieces;        // fp32 operands: the three bf16 pieces of Q, K, V, dO (wide_piece_bytes(d, 4))
  float* part_q;       // partial dQ of split rows (128 x D per tile)
  float* part_kv;      // partial dK, dV of split columns (2 x 128 x D per tile)
  // head_dim 64 / 128 on a plan: the dK/dV walk stores every dS tile here
  // ([BH][nnzb] tiles of 128 x 128 16-bit values, in BSR order, layout in
  // tc_bwd.cu) and the dQ walk sums dS K over them instead of recomputing
  // the scores; null: the dQ walk recomputes them.
  void* dS;
  const int32_t* bsr_of_bsc;  // [nnzb] BSR position of each BSC entry (with dS)
  int nnzb;                   // stored blocks (with dS)
  // head_dim 256 / 512, 16-bit, on a plan: the wide dK walk also stores each
  // P^T tile ([BH][nnzb] in BSC order) and the dV walk streams them
  // (launch_dv_ps) instead of recomputing the scores; null: it recomputes.
  void* dP;
  int* status;
};

// One work item as the planner writes it (see sched.cuh / plan.cu).
struct PlanItem {
  int32_t line;   // block row or block column
  int32_t first;  // offset of its first entry in col_idx / row_idx
  int32_t n;      // stored blocks in the item
  int32_t slot;   // -1: the whole line; else the partial-result slot of this chunk
};

// Layout of one plan in device scratch (int32 units, 16-byte aligned base):
//   header[8]                  items, work-queue counter, split lines, buckets,
//                              CTAs that finished the current launch, pad
//                              (the kernels leave the work-queue counter at G
//                              and the exit count and every arrival counter
//                              at 0 when they finish, so a plan can be reused
//                              launch after launch without running the
//                              planner again)
//   items[cap_items]           PlanItem, longest first
//   buckets[cap_buckets]       PlanBucket, one per item length, longest first
//   slot_line[cap_slots]       split line of each partial slot
//   line_base[cap_lines]       first slot of each split line
//   line_chunks[cap_lines]     chunks of each split line
//   counters[cap_lines*BH*2]   arrivals per (split line, head, column half)
// Bounds: L >= nnzb * BH / G, so split lines <= G / BH and slots < 2 G / BH.
struct PlanBucket {
  int32_t work;   // first work index of the bucket (items before it times BH)
  int32_t start;  // first item of the bucket
  int32_t count;  // items in the bucket (all of one length)
  int32_t len;
};
static_assert(sizeof(PlanBucket) == 16, "a bucket is read as one 16-byte vector");

struct PlanLayout {
  int32_t* header;
  PlanItem* items;
  PlanBucket* buckets;
  int32_t* slot_line;
  int32_t* line_base;
  int32_t* line_chunks;
  int32_t* counters;
  int cap_items, cap_slots, cap_lines, cap_buckets;
};

// max_len: the longest possible line (0: n, the square grids of attention,
// where no line is ever longer than the n blocks a chunk may hold).  With
// longer lines (an SpMM with more block columns than rows) chunks are capped
// at n blocks, which may need up to max_len + n slots and n split lines.
__host__ __device__ inline void plan_caps(int n, int G, int BH, int* items, int* slots, int* lines, int max_len = 0) {
  const bool wide = max_len > n;
  *items = n + 2 * G + 2 + (wide ? max_len + n : 0);
  *slots = 2 * G / BH + 2 + (wide ? max_len + n : 0);
  *lines = G / BH + 2 + (wide ? n : 0);
}

// int32 words one plan occupies (a multiple of 4).
__host__ __device__ inline size_t plan_words(int n, int G, int BH, int max_len = 0) {
  int ci, cs, cl;
  plan_caps(n, G, BH, &ci, &cs, &cl, max_len);
  const int nl = max_len > n ? max_len : n;  // distinct chunk lengths
  size_t w = 8 + 4 * (size_t)ci + 4 * (size_t)(nl + 1) + cs + 2 * (size_t)cl + 2 * (size_t)cl * BH;
  return (w + 3) & ~(size_t)3;
}

__host__ __device__ inline PlanLayout plan_layout(int32_t* base, int n, int G, int BH, int max_len = 0) {
  PlanLayout l;
  plan_caps(n, G, BH, &l.cap_items, &l.cap_slots, &l.cap_lines, max_len);
  l.cap_buckets = (max_len > n ? max_len : n) + 1;
  l.header = base;
  l.items = (PlanItem*)(base + 8);
  l.buckets = (PlanBucket*)(base + 8 + 4 * (size_t)l.cap_items);
  l.slot_line = (int32_t*)(l.buckets + l.cap_buckets);
  l.line_base = l.slot_line + l.cap_slots;
  l.line_chunks = l.line_base + l.cap_lines;
  l.counters = l.line_chunks + l.cap_lines;
  return l;
}

// Partial-result tiles a split plan may need: cap_slots * BH.
__host__ __device__ inline size_t plan_tiles(int n, int G, int BH, int max_len = 0) {
  int ci, cs, cl;
  plan_caps(n, G, BH, &ci, &cs, &cl, max_len);
  return (size_t)cs * BH;
}

struct PlanList {
  const int32_t* ptr;  // [n + 1] prefix offsets (row_ptr or col_ptr)
  int32_t* plan;       // plan_words(n, G, BH) int32 of scratch
};

// The outputs of empty lines (delta.cu): for every line with no stored block
// (ptr[i + 1] == ptr[i]) and every head, the 128 rows of each non-null
// output are zeroed and, when given, row_max = -inf and row_denom = 0.
struct ZeroTarget {
  const int32_t* ptr;  // [nb + 1] line offsets (row_ptr or col_ptr)
  void* out[2];        // [BH * S, D] outputs (null: none)
  float* row_max;      // [BH * S] or null
  float* row_denom;    // [BH * S] or null
};
struct ZeroArgs {
  ZeroTarget t[2];
  int targets;    // 1 or 2
  int nb, BH, S;
  int row_bytes;  // D * element size, a multiple of 16
};
struct PlanArgs {
  PlanList list[3];
  int n;            // lines per list (block rows = block columns)
  int max_len;      // longest possible line (blocks per line; 0: n, the square grids of attention)
  int G;            // persistent CTAs of the kernels that read the plan
  int BH;
  int allow_split;  // 0: every line is one item (no partial results)
  int skip_empty;   // 1: lines with no stored block get no item (their
                    // outputs come from launch_zero_lines, or from the
                    // zero_ctas CTAs below)
  int* status;
  // zero_ctas > 0: the planner launch also writes the outputs of the empty
  // lines of `zero` with that many CTAs (what launch_zero_lines does)
  ZeroArgs zero;
  int zero_ctas;
};

// Builds `lists` (1 to 3) plans.
bsr_status launch_plan(const PlanArgs& p, int lists, cudaStream_t s);
// Delta / lse2 and the plans of `p` in one launch where the plans are small
// (else launch_delta then launch_plan).
bsr_status launch_delta_plan(const BwdArgs& a, const PlanArgs& p, int lists, cudaStream_t s);

// RAII bracket that records a pair of CUDA events around one kernel launch
// when profiling is enabled (bsr_profile_enable).
// Launches `kern` on `s` as a programmatic dependent of the previous kernel
// in the stream: it may start launching while that kernel finishes.  Every
// kernel launched this way calls sm100::griddep_wait() before its first
// access to global memory (the previous kernel may still be reading or
// writing it, including stream-ordered scratch that is reused).
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

// True while per-launch timing is on: kernels that normally overlap on two
// streams then run one after the other, so that each launch's events bracket
// that kernel alone.
bool profiling_launches();

class LaunchTimer {
 public:
  LaunchTimer(const char* name, cudaStream_t stream);
  ~LaunchTimer();

 private:
  int slot_;
  cudaStream_t stream_;
};

// Validates the backward arguments and fills *out (scratch pointers left null).
bsr_status build_bwd_args(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const bsr_tensor* O,
                          const bsr_tensor* dO, const float* row_max, const float* row_denom,
                          const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
                          const int32_t* row_idx, float scale, bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV,
                          BwdArgs* out);

// Backward scratch: a.delta and a.lse2 (BH * S floats each, 16-byte
// aligned), the block-row and block-column plans (plan_words ints each) and,
// with split plans, the partial-result tiles of dQ (128 x D floats each) and
// dK / dV (2 x 128 x D floats each), plan_tiles of each.
size_t bwd_scratch_bytes(const Dims& d, int G, bool split);
// Carves a scratch block of bwd_scratch_bytes at `base` into a's arrays.
void bwd_scratch_carve(BwdArgs* a, void* base, int G, bool split);
// Launches the zero-lines pass (with `zero`: dQ rows of empty block rows,
// dK / dV rows of empty block columns), delta, plan (unless `planned`: the
// plans in a are built, without empty lines), dQ and dK/dV on `s` (scratch
// carved already).
bsr_status run_bwd(const BwdArgs& a, cudaStream_t s, bool split, bool planned, bool zero);

// The forward's argument checks, scratch (its plan, the split rows' partial
// results or the fp32 pieces) and launches (the planner unless `planned`).
bsr_status build_fwd_args(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const int32_t* row_ptr,
                          const int32_t* col_idx, int32_t n_brows, int32_t block, float scale, bsr_tensor* O,
                          float* row_max, float* row_denom, bool two_pass, FwdArgs* out);
size_t fwd_scratch_bytes(const Dims& d, int G);
void fwd_scratch_carve(FwdArgs* a, void* base);
// `zero`: first the zero-lines pass over the empty block rows (the work
// lists leave them out).
bsr_status run_fwd(const FwdArgs& a, cudaStream_t s, bool two_pass, bool planned, bool zero);

// The device status block of the current device (see sm100.cuh wait_limit_ns).
int* status_ptr();

// A second stream of the current device with a fork / join event pair.
// The fork and join must happen while *hold is held (calls from several host
// threads share the pair).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
bsr_status side_stream(SideStream* out, std::unique_lock<std::mutex>* hold);

// Number of SMs of the current device (cached per device); 0 on error.
int sm_count();

// Returns a status for the last launch on this thread (cudaGetLastError).
bsr_status check_launch(const char* what);

// Delta D_i = dO_i . O_i and lse2_i of the backward pass (every dtype and head_dim).
bsr_status launch_delta(const BwdArgs& a, cudaStream_t s);

bsr_status launch_zero_lines(const ZeroArgs& z, cudaStream_t s);

// Tensor-core (tcgen05 / TMA) kernels for bf16 / fp16 operands with head_dim
// 64 / 128; a.plan and a.part must hold the block-row plan built by
// launch_plan and its partial-result tiles.
bool tc_fwd_supported(const Dims& d);
// head_dim 64 / 128, P in TMEM.  pass 0: the online-softmax forward; 1 and
// 2: the statistics pass and then the output pass of the statistics-first
// variant (the output pass reads the row_max / row_denom the first wrote).
bsr_status launch_fwd_tc2(const FwdArgs& a, cudaStream_t s, int pass = 0);
bool tc_bwd_supported(const Dims& d);

// Tensor-core kernels for the other cases (tc_wide.cu): bf16 / fp16 with
// head_dim 256 / 512 and fp32 with any head_dim, on plans built with
// plan_heads(d) heads (split plans need part_tile_bytes per partial tile:
// the forward's a.part, the backward's part_q and, for dV then dK, two sets
// at part_kv).  fp32 operands need wide_piece_bytes(d, tensors) of scratch
// in a.pieces for their bf16 pieces.
bool wide_supported(const Dims& d);
size_t wide_piece_bytes(const Dims& d, int tensors);
// Heads the planner is given for d's kernels: BH for the head_dim 64 / 128
// tensor-core kernels; for the wide kernels BH times the output slices of
// head_dim each work item covers (each slice is planned as a head of its
// own, so its chunks of a split line merge on their own counter).
int plan_heads(const Dims& d);
// Bytes of one partial-result tile of a split line, forward or backward
// (the forward's carries the chunk's row statistics).
size_t part_tile_bytes(const Dims& d, bool fwd);
bsr_status launch_fwd_wide(const FwdArgs& a, cudaStream_t s);
// dQ on the row plan, dV on col_plan, dK on col_plan2, after launch_delta.
bsr_status launch_bwd_wide(const BwdArgs& a, cudaStream_t s);

// Y = A X for a BSR matrix A of 128 x 128 blocks, and the walk of the
// screened product over its kept tiles (tc_spmm.cu).
struct SpmmArgs {
  const void* A;            // stored blocks, [nnzb][128][128] row-major (screened: the dense [n][n] A)
  const void* X;            // [n_bcols * 128][n_cols] row-major
  void* Y;                  // [n_brows * 128][n_cols] row-major
  const int32_t* row_ptr;   // [n_brows + 1]
  const int32_t* col_idx;   // [nnzb]
  int n_brows, n_bcols, nnzb, n_cols;
  int dtype;                // BSR_BF16 or BSR_F16
  int* status;
  int32_t* plan;            // set by the launcher: the rows' work list (column tiles as heads)
  float* part;              // set by the launcher: partial products of split rows
  const int32_t* cls;       // screened: per listed tile, 1 = kept whole, 2 = masked element by element
  const float* diag;        // screened: the bounds' diagonal
  float t;                  // screened: sqrt(threshold)
};
bsr_status launch_spmm_tc(const SpmmArgs& a, cudaStream_t s);

// The screened product's tile list (plan.cu): every 128 x 128 tile (m, k) of
// A classified by the least and largest bound q = sqrt(|diag|) of its rows
// and columns (skipped, kept whole, masked element by element), the kept
// tiles of each block row listed in BSR form with their class.
enum : int { kTileSkip = 0, kTileFull = 1, kTilePartial = 2, kScreenMaxBlocks = 512 };
struct ScreenListArgs {
  const float* diag;
  int nb;            // n / 128 <= kScreenMaxBlocks
  float t;           // sqrt(threshold)
  int32_t* row_ptr;  // [nb + 1]
  int32_t* col_idx;  // [nb * nb]
  int32_t* cls;      // [nb * nb]
};
// Builds the tile list and then plan p (one list, over l.row_ptr) in one launch.
bsr_status launch_screen_plan(const ScreenListArgs& l, const PlanArgs& p, cudaStream_t s);

// C = (A o M) B with M[i, j] = (sqrt|diag_i| sqrt|diag_j| > sqrt(threshold)) (tc_screened.cu).
struct ScreenedArgs {
  const void* A;       // [n][n] row-major
  const float* diag;   // [n]
  const void* B;       // [n][n_cols] row-major
  void* C;             // [n][n_cols] row-major
  int n, n_cols;
  float threshold;
  int dtype;           // BSR_BF16 or BSR_F16
  int* status;
};
bsr_status launch_screened_tc(const ScreenedArgs& a, cudaStream_t s);
// Persistent grid of the tensor-core kernels: min(SMs, lines * BH); 0 on error.
int tc_grid(const Dims& d);
// Bytes of one forward partial-result tile (split rows), head_dim 64 / 128.
size_t fwd_part_bytes(int D);
bsr_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s);
// The dQ walk over stored dS tiles (a.dS, a.nnzb) for 16-bit operands with
// head_dim 256 / 512, on the wide kernels' block-row plan (a.row_plan,
// plan_heads(d) heads, partial tiles at a.part_q), after the dK walk that
// stored the tiles.
bsr_status launch_dq_ds(const BwdArgs& a, cudaStream_t s);
// dV_n = sum_m P^T_nm dO_m over stored P^T tiles (a.dP) for 16-bit operands
// with head_dim 256 / 512, on the wide kernels' dV plan (a.col_plan, partial
// tiles at a.part_kv), after the dK walk that stored the tiles.
bsr_status launch_dv_ps(const BwdArgs& a, cudaStream_t s);

}  // namespace bsr
