// Reusable plans: the work lists of one block mask built once and kept, with
// every scratch array the forward and backward passes need, so that a call
// on a plan launches only the attention kernels (and the backward's delta
// pass): no planner, no allocation.  The pages build their kernels once per
// static structure and reuse them call after call ("trnsparse 0.7.0 ->
// 0.9.0" diff, CHANGELOG [0.8.0], static structure); here the structure is
// data, so what is built once is the work lists over it.
//
// A plan owns one cudaMalloc block:
//   copies of row_ptr, col_idx, col_ptr, row_idx (16-byte aligned each)
//   the block-row plan (forward and dQ), two block-column plans (dK / dV;
//     the wide kernels' dV and dK walks)
//   the forward's split-line partial tiles and the backward's
//   the bf16 pieces of fp32 operands (wide kernels)
//   delta and lse2 (one fp32 value each per query row)
//   the BSR position of each BSC entry
// and, in a second cudaMalloc block, the dS tiles the dK/dV (or dK) walk
// stores for the dQ walk (batch * heads * nnzb tiles of 32 KB, 64 KB for
// fp32 operands; without that memory the plan's dQ walk recomputes the
// scores instead).
// The kernels put the plans' work-queue counters back to the grid size and
// their arrival counters back to 0 when they finish, so the lists are built
// once, at creation.

#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <vector>

#include "kernels.h"

struct bsr_plan_s {
  int device;
  int batch, heads, seq, head_dim, dtype;
  int nb, nnzb, G;
  int empty_rows, empty_cols;  // block rows / columns with no stored block
  void* mem;
  int32_t *row_ptr, *col_idx, *col_ptr, *row_idx;
  int32_t *row_plan, *col_plan, *col_plan2;
  float *fwd_part, *part_q, *part_kv, *delta, *lse2;
  void* pieces;
  int32_t* bsr_of_bsc;  // null unless dS is set
  void* dS;             // own cudaMalloc block, or null
  void* dP;             // in the dS block (the wide kernels' operands), or null
};

namespace bsr {
namespace {

size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

bsr_status plan_matches(const bsr_plan* plan, const bsr_tensor* Q, const char* who) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: cudaGetDevice failed", who);
  if (dev != plan->device)
    return fail(BSR_ERR_INVALID_ARG, "%s: the plan was built on device %d, the current device is %d", who,
                plan->device, dev);
  if (Q->batch != plan->batch || Q->heads != plan->heads || Q->seq != plan->seq || Q->head_dim != plan->head_dim ||
      Q->dtype != plan->dtype)
    return fail(BSR_ERR_INVALID_ARG,
                "%s: operands [%d, %d, %d, %d] dtype %d differ from the plan's [%d, %d, %d, %d] dtype %d", who,
                Q->batch, Q->heads, Q->seq, Q->head_dim, Q->dtype, plan->batch, plan->heads, plan->seq,
                plan->head_dim, plan->dtype);
  return BSR_OK;
}

}  // namespace
}  // namespace bsr

using namespace bsr;

extern "C" bsr_status bsr_plan_create(const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
                                      const int32_t* row_idx, int32_t n_brows, int32_t batch, int32_t heads,
                                      int32_t head_dim, int32_t dtype, void* stream, bsr_plan** out) {
  if (!out) return fail(BSR_ERR_INVALID_ARG, "bsr_plan_create: null output handle");
  *out = nullptr;
  if (!row_ptr || !col_idx || !col_ptr || !row_idx)
    return fail(BSR_ERR_INVALID_ARG, "bsr_plan_create: null structure array");
  if (n_brows < 1 || batch < 1 || heads < 1 || (long long)n_brows * 128 > (1LL << 30) ||
      (long long)batch * heads > (1LL << 30))
    return fail(BSR_ERR_INVALID_ARG, "bsr_plan_create: sizes n_brows %d, batch %d, heads %d", n_brows, batch, heads);
  if (dtype != BSR_F32 && dtype != BSR_BF16 && dtype != BSR_F16)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_plan_create: dtype %d not supported", dtype);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 && head_dim != 512)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_plan_create: head_dim %d not supported (64, 128, 256 or 512)", head_dim);
  Dims d{};
  d.BH = batch * heads;
  d.S = n_brows * 128;
  d.D = head_dim;
  d.nb = n_brows;
  d.dtype = dtype;
  d.scale = 1.f;
  if (!tc_bwd_supported(d) && !wide_supported(d))
    return fail(BSR_ERR_UNSUPPORTED, "bsr_plan_create: dtype %d with head_dim %d", dtype, head_dim);
  int* status = status_ptr();
  if (!status) return fail(BSR_ERR_CUDA, "bsr_plan_create: no CUDA device");
  const int G = tc_grid(d);
  if (G <= 0) return fail(BSR_ERR_CUDA, "bsr_plan_create: cannot query the SM count");
  cudaStream_t s = (cudaStream_t)stream;
  // the number of stored blocks, from both pointer arrays, and the empty
  // lines (no stored block), whose outputs the zero-lines pass writes
  std::vector<int32_t> rp(n_brows + 1), cp(n_brows + 1);
  cudaError_t e = cudaMemcpyAsync(rp.data(), row_ptr, sizeof(int32_t) * (n_brows + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cp.data(), col_ptr, sizeof(int32_t) * (n_brows + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_plan_create: reading the offsets: %s", cudaGetErrorString(e));
  const int nnzb = rp[n_brows];
  if (nnzb < 0 || (long long)nnzb > (long long)n_brows * n_brows || cp[n_brows] != nnzb)
    return fail(BSR_ERR_INVALID_ARG, "bsr_plan_create: row_ptr[n_brows] = %d and col_ptr[n_brows] = %d",
                rp[n_brows], cp[n_brows]);
  int empty_rows = 0, empty_cols = 0;
  for (int i = 0; i < n_brows; ++i) {
    empty_rows += rp[i + 1] == rp[i] ? 1 : 0;
    empty_cols += cp[i + 1] == cp[i] ? 1 : 0;
  }
  // the dK/dV (or dK) walk hands its dS tiles to the dQ walk, stored by BSR
  // position; map each BSC entry to it
  std::vector<int32_t> bsr_of_bsc;
  // a block's dS: one 16-bit tile, or two bf16 piece tiles for fp32 operands
  const size_t ds_tile_b = d.dtype == BSR_F32 ? 2 * 128 * 128 * 2 : 128 * 128 * 2;
  const bool want_ds = nnzb > 0 && (size_t)d.BH * (size_t)nnzb <= ((size_t)1 << 62) / ds_tile_b;
  // the wide kernels (16-bit at head_dim 256 / 512, fp32): the dK walk also
  // stores P^T for a streaming dV walk (the head_dim-64 / 128 dK/dV walk
  // computes dV itself)
  const bool want_dp = want_ds && !tc_bwd_supported(d);
  if (want_ds) {
    std::vector<int32_t> ci(nnzb), ri(nnzb);
    e = cudaMemcpyAsync(ci.data(), col_idx, sizeof(int32_t) * nnzb, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ri.data(), row_idx, sizeof(int32_t) * nnzb, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_plan_create: reading the indices: %s", cudaGetErrorString(e));
    std::vector<int64_t> key(nnzb);
    std::vector<int32_t> ord(nnzb);
    for (int m = 0; m < n_brows; ++m)
      for (int j = rp[m]; j < rp[m + 1]; ++j) key[j] = (int64_t)m * n_brows + ci[j];
    for (int j = 0; j < nnzb; ++j) ord[j] = j;
    std::sort(ord.begin(), ord.end(), [&](int32_t x, int32_t y) { return key[x] < key[y]; });
    bsr_of_bsc.resize(nnzb);
    for (int n = 0; n < n_brows; ++n) {
      for (int q = cp[n]; q < cp[n + 1]; ++q) {
        const int m = ri[q];
        const int64_t want = (int64_t)m * n_brows + n;
        auto it = std::lower_bound(ord.begin(), ord.end(), want,
                                   [&](int32_t x, int64_t v) { return key[x] < v; });
        if (m < 0 || m >= n_brows || it == ord.end() || key[*it] != want)
          return fail(BSR_ERR_INVALID_ARG,
                      "bsr_plan_create: BSC entry %d (block row %d, column %d) is not a stored block of the BSR arrays",
                      q, m, n);
        bsr_of_bsc[q] = *it;
      }
    }
  }

  const int pheads = plan_heads(d);
  const size_t pw = plan_words(d.nb, G, pheads);
  const size_t tiles = plan_tiles(d.nb, G, pheads);
  const size_t rows = (size_t)d.BH * d.S;
  const size_t ptr_b = align16(sizeof(int32_t) * (n_brows + 1));
  const size_t idx_b = align16(sizeof(int32_t) * (nnzb > 0 ? nnzb : 1));
  const size_t plans_b = 3 * sizeof(int32_t) * pw;  // a multiple of 16 (plan_words is a multiple of 4)
  const size_t fpart_b = align16(part_tile_bytes(d, true) * tiles);
  const size_t bset_b = part_tile_bytes(d, false) * tiles;  // one set: dQ, dV or dK (a multiple of 16)
  const size_t bpart_b = 3 * bset_b;
  const size_t stat_b = 2 * align16(sizeof(float) * rows);
  const size_t piece_b = wide_piece_bytes(d, 4);
  const size_t map_b = want_ds ? idx_b : 0;
  const size_t total = 2 * ptr_b + 2 * idx_b + plans_b + fpart_b + bpart_b + stat_b + piece_b + map_b;

  bsr_plan* p = new (std::nothrow) bsr_plan();
  if (!p) return fail(BSR_ERR_INVALID_ARG, "bsr_plan_create: out of host memory");
  if ((e = cudaGetDevice(&p->device)) != cudaSuccess || (e = cudaMalloc(&p->mem, total)) != cudaSuccess) {
    delete p;
    return fail(BSR_ERR_CUDA, "bsr_plan_create: cudaMalloc(%zu): %s", total, cudaGetErrorString(e));
  }
  p->batch = batch;
  p->heads = heads;
  p->seq = d.S;
  p->head_dim = head_dim;
  p->dtype = dtype;
  p->nb = n_brows;
  p->nnzb = nnzb;
  p->empty_rows = empty_rows;
  p->empty_cols = empty_cols;
  p->G = G;
  char* c = (char*)p->mem;
  p->row_ptr = (int32_t*)c;
  c += ptr_b;
  p->col_ptr = (int32_t*)c;
  c += ptr_b;
  p->col_idx = (int32_t*)c;
  c += idx_b;
  p->row_idx = (int32_t*)c;
  c += idx_b;
  p->row_plan = (int32_t*)c;
  p->col_plan = p->row_plan + pw;
  p->col_plan2 = p->col_plan + pw;
  c += plans_b;
  p->fwd_part = (float*)c;
  c += fpart_b;
  p->part_q = (float*)c;
  p->part_kv = (float*)(c + bset_b);
  c += bpart_b;
  p->delta = (float*)c;
  p->lse2 = (float*)(c + align16(sizeof(float) * rows));
  c += stat_b;
  p->pieces = piece_b ? (void*)c : nullptr;
  c += piece_b;
  p->bsr_of_bsc = nullptr;
  p->dS = nullptr;
  p->dP = nullptr;
  if (want_ds) {
    void* ds = nullptr;
    const size_t ds_b = (size_t)d.BH * nnzb * ds_tile_b;
    if (cudaMalloc(&ds, want_dp ? 2 * ds_b : ds_b) == cudaSuccess) {
      p->dS = ds;
      p->dP = want_dp ? (void*)((char*)ds + ds_b) : nullptr;
      p->bsr_of_bsc = (int32_t*)c;
    } else {
      cudaGetLastError();  // out of memory: the dQ walk recomputes the scores
    }
  }

  e = cudaMemcpyAsync(p->row_ptr, row_ptr, sizeof(int32_t) * (n_brows + 1), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->col_ptr, col_ptr, sizeof(int32_t) * (n_brows + 1), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && nnzb > 0)
    e = cudaMemcpyAsync(p->col_idx, col_idx, sizeof(int32_t) * nnzb, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && nnzb > 0)
    e = cudaMemcpyAsync(p->row_idx, row_idx, sizeof(int32_t) * nnzb, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && p->dS) {
    e = cudaMemcpyAsync(p->bsr_of_bsc, bsr_of_bsc.data(), sizeof(int32_t) * nnzb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the host vector goes out of scope
  }
  if (e != cudaSuccess) {
    if (p->dS) cudaFree(p->dS);
    cudaFree(p->mem);
    delete p;
    return fail(BSR_ERR_CUDA, "bsr_plan_create: copying the structure: %s", cudaGetErrorString(e));
  }
  PlanArgs pa{};
  pa.list[0] = PlanList{p->row_ptr, p->row_plan};
  pa.list[1] = PlanList{p->col_ptr, p->col_plan};
  pa.list[2] = PlanList{p->col_ptr, p->col_plan2};
  pa.n = d.nb;
  pa.G = G;
  pa.BH = pheads;
  pa.allow_split = 1;
  pa.skip_empty = 1;
  pa.status = status;
  bsr_status st = launch_plan(pa, 3, s);
  if (st != BSR_OK) {
    cudaStreamSynchronize(s);
    if (p->dS) cudaFree(p->dS);
    cudaFree(p->mem);
    delete p;
    return st;
  }
  *out = p;
  return BSR_OK;
}

extern "C" bsr_status bsr_plan_destroy(bsr_plan* plan) {
  if (!plan) return BSR_OK;
  cudaError_t e = plan->dS ? cudaFree(plan->dS) : cudaSuccess;
  const cudaError_t e2 = cudaFree(plan->mem);
  if (e == cudaSuccess) e = e2;
  delete plan;
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_plan_destroy: cudaFree: %s", cudaGetErrorString(e));
  return BSR_OK;
}

extern "C" bsr_status bsr_attn_fwd_plan(const bsr_plan* plan, const bsr_tensor* Q, const bsr_tensor* K,
                                        const bsr_tensor* V, float scale, bsr_tensor* O, float* row_max,
                                        float* row_denom, void* stream) {
  if (!plan) return fail(BSR_ERR_INVALID_ARG, "bsr_attn_fwd_plan: null plan");
  FwdArgs a{};
  bsr_status st = build_fwd_args(Q, K, V, plan->row_ptr, plan->col_idx, plan->nb, 128, scale, O, row_max, row_denom,
                                 false, &a);
  if (st != BSR_OK) return st;
  if ((st = plan_matches(plan, Q, "bsr_attn_fwd_plan")) != BSR_OK) return st;
  if (a.G != plan->G) return fail(BSR_ERR_INVALID_ARG, "bsr_attn_fwd_plan: the plan was built for another grid");
  a.plan = plan->row_plan;
  a.part = plan->fwd_part;
  a.pieces = plan->pieces;
  return run_fwd(a, (cudaStream_t)stream, false, true, plan->empty_rows > 0);
}

extern "C" bsr_status bsr_attn_bwd_plan(const bsr_plan* plan, const bsr_tensor* Q, const bsr_tensor* K,
                                        const bsr_tensor* V, const bsr_tensor* O, const bsr_tensor* dO,
                                        const float* row_max, const float* row_denom, float scale, bsr_tensor* dQ,
                                        bsr_tensor* dK, bsr_tensor* dV, void* stream) {
  if (!plan) return fail(BSR_ERR_INVALID_ARG, "bsr_attn_bwd_plan: null plan");
  BwdArgs a{};
  bsr_status st = build_bwd_args(Q, K, V, O, dO, row_max, row_denom, plan->row_ptr, plan->col_idx, plan->col_ptr,
                                 plan->row_idx, scale, dQ, dK, dV, &a);
  if (st != BSR_OK) return st;
  if ((st = plan_matches(plan, Q, "bsr_attn_bwd_plan")) != BSR_OK) return st;
  if (tc_grid(a.d) != plan->G) return fail(BSR_ERR_INVALID_ARG, "bsr_attn_bwd_plan: the plan was built for another grid");
  a.delta = plan->delta;
  a.lse2 = plan->lse2;
  a.row_plan = plan->row_plan;
  a.col_plan = plan->col_plan;
  a.col_plan2 = plan->col_plan2;
  a.part_q = plan->part_q;
  a.part_kv = plan->part_kv;
  a.pieces = plan->pieces;
  a.dS = plan->dS;
  a.dP = plan->dP;
  a.bsr_of_bsc = plan->bsr_of_bsc;
  a.nnzb = plan->nnzb;
  return run_bwd(a, (cudaStream_t)stream, true, true, plan->empty_rows + plan->empty_cols > 0);
}

extern "C" bsr_status bsr_plan_work_list(const bsr_plan* plan, int32_t list, int32_t* items, int32_t cap,
                                         int32_t* info, void* stream) {
  if (!plan || !items || !info) return fail(BSR_ERR_INVALID_ARG, "bsr_plan_work_list: null argument");
  if (list < 0 || list > 2) return fail(BSR_ERR_INVALID_ARG, "bsr_plan_work_list: list %d (0, 1 or 2)", list);
  Dims d{};
  d.BH = plan->batch * plan->heads;
  d.S = plan->seq;
  d.D = plan->head_dim;
  d.nb = plan->nb;
  d.dtype = plan->dtype;
  const int heads = plan_heads(d);
  int32_t* base = list == 0 ? plan->row_plan : (list == 1 ? plan->col_plan : plan->col_plan2);
  const PlanLayout lay = plan_layout(base, plan->nb, plan->G, heads);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t header[8];
  cudaError_t e = cudaMemcpyAsync(header, lay.header, sizeof(header), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_plan_work_list: %s", cudaGetErrorString(e));
  const int n = header[0];
  if (n < 0 || n > lay.cap_items) return fail(BSR_ERR_DEVICE_CHECK, "bsr_plan_work_list: %d items in the plan", n);
  if (n > cap) return fail(BSR_ERR_INVALID_ARG, "bsr_plan_work_list: %d items do not fit %d", n, cap);
  static_assert(sizeof(PlanItem) == 4 * sizeof(int32_t), "an item is four int32");
  if (n > 0) {
    e = cudaMemcpyAsync(items, lay.items, sizeof(PlanItem) * (size_t)n, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_plan_work_list: %s", cudaGetErrorString(e));
  }
  info[0] = n;
  info[1] = plan->G;
  info[2] = heads;
  info[3] = header[3];  // buckets (distinct item lengths)
  return BSR_OK;
}
