// C-ABI front end: argument checks, scratch, the device status word, kernel
// timing and dispatch to the attention kernels.

#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"

namespace bsr {

namespace {
thread_local std::string g_error;

// Device status block (see wait_limit_ns in sm100.cuh): word 0 is the
// status word, set by kernels whose bounded waits give up or whose index
// checks fail and read and cleared by bsr_attn_check; words 2..3 hold the
// bounded waits' limit in nanoseconds (2 s; bsr_set_wait_limit changes it).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
__device__ __align__(16) int g_status[4] = {0, 0, (int)kDefaultWaitLimitNs, 0};

}  // namespace

int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static std::mutex mu;
  static std::vector<int*> cache;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, nullptr);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    cache[dev] = (int*)p;
  }
  return cache[dev];
}

namespace {

// ------------------------------------------------------------ profiling --
struct TimedLaunch {
  std::string name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<TimedLaunch> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

bsr_status fail(bsr_status status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return status;
}

bool profiling_launches() {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  return g_prof_on;
}

LaunchTimer::LaunchTimer(const char* name, cudaStream_t stream) : slot_(-1), stream_(stream) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on) return;
  TimedLaunch t{name, take_event(), take_event()};
  cudaEventRecord(t.start, stream);
  g_prof.push_back(t);
  slot_ = (int)g_prof.size() - 1;
}

LaunchTimer::~LaunchTimer() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (slot_ < (int)g_prof.size()) cudaEventRecord(g_prof[slot_].stop, stream_);
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (!cache[dev] && cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    cache[dev] = 0;
  return cache[dev];
}

// Per device: a second stream and a fork / join event pair, for kernels of
// one call that may run side by side (created once, kept for the process).
bsr_status side_stream(SideStream* out, std::unique_lock<std::mutex>* hold) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(BSR_ERR_CUDA, "side stream: cudaGetDevice failed");
  static std::mutex mu;
  static std::vector<SideStream> cache;
  std::unique_lock<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1);
  SideStream& ss = cache[dev];
  if (!ss.s) {
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess)
      return fail(BSR_ERR_CUDA, "side stream: create failed: %s", cudaGetErrorString(cudaGetLastError()));
    ss.s = st;
    ss.fork = f;
    ss.join = j;
  }
  *out = ss;
  *hold = std::move(lock);  // the caller forks and joins under the lock
  return BSR_OK;
}

bsr_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return BSR_OK;
}

namespace {

bsr_status check_tensor(const bsr_tensor* t, const char* name, const bsr_tensor* ref) {
  if (!t) return fail(BSR_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (!t->data) return fail(BSR_ERR_INVALID_ARG, "%s: null data pointer", name);
  if ((uintptr_t)t->data & 15) return fail(BSR_ERR_INVALID_ARG, "%s: data pointer is not 16-byte aligned", name);
  if (t->dtype != BSR_F32 && t->dtype != BSR_BF16 && t->dtype != BSR_F16)
    return fail(BSR_ERR_UNSUPPORTED, "%s: dtype %d not supported (BSR_F32, BSR_BF16 or BSR_F16)", name, t->dtype);
  if (t->batch < 1 || t->heads < 1 || t->seq < 1)
    return fail(BSR_ERR_INVALID_ARG, "%s: non-positive shape [%d, %d, %d, %d]", name, t->batch, t->heads, t->seq,
                t->head_dim);
  if (t->head_dim != 64 && t->head_dim != 128 && t->head_dim != 256 && t->head_dim != 512)
    return fail(BSR_ERR_UNSUPPORTED, "%s: head_dim %d not supported (64, 128, 256 or 512)", name, t->head_dim);
  if (ref && (t->batch != ref->batch || t->heads != ref->heads || t->seq != ref->seq || t->head_dim != ref->head_dim))
    return fail(BSR_ERR_INVALID_ARG, "%s: shape [%d, %d, %d, %d] differs from Q [%d, %d, %d, %d]", name, t->batch,
                t->heads, t->seq, t->head_dim, ref->batch, ref->heads, ref->seq, ref->head_dim);
  if (ref && t->dtype != ref->dtype)
    return fail(BSR_ERR_UNSUPPORTED, "%s: dtype %d differs from Q's %d (mixed operands are not converted)", name,
                t->dtype, ref->dtype);
  return BSR_OK;
}

bsr_status make_dims(const bsr_tensor* Q, float scale, Dims* d) {
  if ((long long)Q->batch * Q->heads > (1LL << 30))
    return fail(BSR_ERR_INVALID_ARG, "batch * heads = %lld too large", (long long)Q->batch * Q->heads);
  if (Q->seq % 128 != 0) return fail(BSR_ERR_INVALID_ARG, "seq %d is not a multiple of the block size 128", Q->seq);
  if (!isfinite(scale)) return fail(BSR_ERR_INVALID_ARG, "scale is not finite");
  d->BH = Q->batch * Q->heads;
  d->S = Q->seq;
  d->D = Q->head_dim;
  d->nb = Q->seq / 128;
  d->dtype = Q->dtype;
  d->scale = scale;
  return BSR_OK;
}

}  // namespace
}  // namespace bsr

using namespace bsr;

extern "C" const char* bsr_last_error(void) { return g_error.c_str(); }

namespace bsr {

bsr_status build_fwd_args(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const int32_t* row_ptr,
                          const int32_t* col_idx, int32_t n_brows, int32_t block, float scale, bsr_tensor* O,
                          float* row_max, float* row_denom, bool two_pass, FwdArgs* out) {
  bsr_status st;
  if (block != 128) return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_fwd: block %d not supported (128)", block);
  if ((st = check_tensor(Q, "Q", nullptr)) || (st = check_tensor(K, "K", Q)) || (st = check_tensor(V, "V", Q)) ||
      (st = check_tensor(O, "O", Q)))
    return st;
  if (!row_ptr || !col_idx || !row_max || !row_denom)
    return fail(BSR_ERR_INVALID_ARG, "bsr_attn_fwd: null row_ptr / col_idx / row_max / row_denom");
  FwdArgs a{};
  if ((st = make_dims(Q, scale, &a.d))) return st;
  if (n_brows != a.d.nb)
    return fail(BSR_ERR_INVALID_ARG, "bsr_attn_fwd: n_brows %d but seq %d / 128 = %d", n_brows, Q->seq, a.d.nb);
  a.Q = Q->data;
  a.K = K->data;
  a.V = V->data;
  a.O = O->data;
  a.row_max = row_max;
  a.row_denom = row_denom;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  if (two_pass && !tc_fwd_supported(a.d))
    return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_fwd_two_pass: bf16 / fp16 operands with head_dim 64 or 128 only");
  // bf16 / fp16 with head_dim 64 / 128: the key-halves kernel (tc_fwd2.cu),
  // which splits long rows; everything else: the wide kernel (tc_wide.cu)
  if (!tc_fwd_supported(a.d) && !wide_supported(a.d))
    return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_fwd: dtype %d with head_dim %d", a.d.dtype, a.d.D);
  a.status = status_ptr();
  if (!a.status) return fail(BSR_ERR_CUDA, "bsr_attn_fwd: no CUDA device");
  a.G = tc_grid(a.d);
  if (a.G <= 0) return fail(BSR_ERR_CUDA, "bsr_attn_fwd: cannot query the SM count");
  *out = a;
  return BSR_OK;
}

size_t fwd_scratch_bytes(const Dims& d, int G) {
  const int heads = plan_heads(d);
  size_t bytes = sizeof(int32_t) * plan_words(d.nb, G, heads);
  bytes += part_tile_bytes(d, true) * plan_tiles(d.nb, G, heads);
  if (!tc_fwd_supported(d)) bytes += wide_piece_bytes(d, 3);
  return bytes;
}

void fwd_scratch_carve(FwdArgs* a, void* base) {
  const int heads = plan_heads(a->d);
  char* p = (char*)base;
  a->plan = (int32_t*)p;
  p += sizeof(int32_t) * plan_words(a->d.nb, a->G, heads);
  a->part = (float*)p;
  p += part_tile_bytes(a->d, true) * plan_tiles(a->d.nb, a->G, heads);  // a multiple of 16 bytes
  a->pieces = tc_fwd_supported(a->d) ? nullptr : (void*)p;
}

// CTAs for the zero pass when it rides in a planner launch: one per
// (target, line, head) triple up to one per SM (most lines are not empty,
// and a CTA checks a line with two loads).
static int zero_ctas(const ZeroArgs& z) {
  const long long triples = (long long)z.targets * z.nb * z.BH;
  const int sms = sm_count();
  const long long cap = sms > 0 ? sms : 1;
  return (int)(triples < cap ? (triples > 0 ? triples : 1) : cap);
}

// The forward pass on carved scratch: the planner first unless the plan in
// a.plan is already built (a bsr_plan), then the online-softmax pass, or
// (two_pass) the statistics pass and then the output pass of the
// statistics-first variant.  The kernels leave the plan's counters at 0, so
// both passes run on one plan.  The work lists leave out empty block rows;
// with `zero` their outputs (zero rows, row_max -inf, row_denom 0) come from
// the zero-lines pass.
bsr_status run_fwd(const FwdArgs& a, cudaStream_t s, bool two_pass, bool planned, bool zero) {
  bsr_status st = BSR_OK;
  const bool tc2 = tc_fwd_supported(a.d);
  ZeroArgs z{};
  if (zero) {
    z.t[0] = ZeroTarget{a.row_ptr, {a.O, nullptr}, a.row_max, a.row_denom};
    z.targets = 1;
    z.nb = a.d.nb;
    z.BH = a.d.BH;
    z.S = a.d.S;
    z.row_bytes = a.d.D * (a.d.dtype == BSR_F32 ? 4 : 2);
    // on a plan the zero pass has a launch of its own; otherwise it rides in
    // the planner's launch
    if (planned && (st = launch_zero_lines(z, s)) != BSR_OK) return st;
  }
  if (!planned) {
    PlanArgs p{};
    p.list[0] = PlanList{a.row_ptr, a.plan};
    p.n = a.d.nb;
    p.G = a.G;
    p.BH = plan_heads(a.d);
    p.allow_split = 1;
    p.skip_empty = 1;
    p.status = a.status;
    if (zero) {
      p.zero = z;
      p.zero_ctas = zero_ctas(z);
    }
    if ((st = launch_plan(p, 1, s)) != BSR_OK) return st;
  }
  if (!tc2) return launch_fwd_wide(a, s);
  if (!two_pass) return launch_fwd_tc2(a, s, 0);
  if ((st = launch_fwd_tc2(a, s, 1)) != BSR_OK) return st;
  return launch_fwd_tc2(a, s, 2);
}

namespace {

bsr_status fwd_impl(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const int32_t* row_ptr,
                    const int32_t* col_idx, int32_t n_brows, int32_t block, float scale, bsr_tensor* O,
                    float* row_max, float* row_denom, void* stream, bool two_pass) {
  FwdArgs a{};
  bsr_status st = build_fwd_args(Q, K, V, row_ptr, col_idx, n_brows, block, scale, O, row_max, row_denom, two_pass, &a);
  if (st != BSR_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, fwd_scratch_bytes(a.d, a.G), s);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_attn_fwd: cudaMallocAsync: %s", cudaGetErrorString(e));
  fwd_scratch_carve(&a, scratch);
  st = run_fwd(a, s, two_pass, false, true);
  e = cudaFreeAsync(scratch, s);
  if (st == BSR_OK && e != cudaSuccess) st = fail(BSR_ERR_CUDA, "bsr_attn_fwd: cudaFreeAsync: %s", cudaGetErrorString(e));
  return st;
}

}  // namespace
}  // namespace bsr

extern "C" bsr_status bsr_attn_fwd(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                                   const int32_t* row_ptr, const int32_t* col_idx, int32_t n_brows,
                                   int32_t block, float scale,
                                   bsr_tensor* O, float* row_max, float* row_denom, void* stream) {
  return bsr::fwd_impl(Q, K, V, row_ptr, col_idx, n_brows, block, scale, O, row_max, row_denom, stream, false);
}

extern "C" bsr_status bsr_spmm(const void* blocks, int32_t dtype, const int32_t* row_ptr, const int32_t* col_idx,
                               int32_t n_brows, int32_t n_bcols, int32_t nnzb, int32_t block, const void* X,
                               int32_t n_cols, void* Y, void* stream) {
  if (block != 128) return fail(BSR_ERR_UNSUPPORTED, "bsr_spmm: block %d not supported (128)", block);
  if (dtype != BSR_BF16 && dtype != BSR_F16)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_spmm: dtype %d not supported (BSR_BF16 or BSR_F16)", dtype);
  if (n_brows < 1 || n_bcols < 1 || nnzb < 0 || n_cols < 1)
    return fail(BSR_ERR_INVALID_ARG, "bsr_spmm: sizes n_brows %d, n_bcols %d, nnzb %d, n_cols %d", n_brows, n_bcols,
                nnzb, n_cols);
  if (n_cols % 64 != 0) return fail(BSR_ERR_UNSUPPORTED, "bsr_spmm: n_cols %d is not a multiple of 64", n_cols);
  if ((long long)n_bcols * 128 > INT32_MAX || (long long)nnzb * 128 > INT32_MAX || (long long)n_brows * 128 > INT32_MAX)
    return fail(BSR_ERR_INVALID_ARG, "bsr_spmm: too many rows");
  if (!row_ptr || !col_idx || !X || !Y || (nnzb > 0 && !blocks))
    return fail(BSR_ERR_INVALID_ARG, "bsr_spmm: null pointer");
  if ((((uintptr_t)Y) | ((uintptr_t)X) | ((uintptr_t)blocks)) & 15)
    return fail(BSR_ERR_INVALID_ARG, "bsr_spmm: data pointer is not 16-byte aligned");
  SpmmArgs a{};
  a.A = blocks;
  a.X = X;
  a.Y = Y;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.n_brows = n_brows;
  a.n_bcols = n_bcols;
  a.nnzb = nnzb;
  a.n_cols = n_cols;
  a.dtype = dtype;
  a.status = status_ptr();
  if (!a.status) return fail(BSR_ERR_CUDA, "bsr_spmm: no CUDA device");
  cudaStream_t s = (cudaStream_t)stream;
  if (nnzb == 0) {  // no stored block: Y = 0
    const cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)n_brows * 128 * (size_t)n_cols * 2, s);
    return e == cudaSuccess ? BSR_OK : fail(BSR_ERR_CUDA, "bsr_spmm: cudaMemsetAsync: %s", cudaGetErrorString(e));
  }
  return launch_spmm_tc(a, s);
}

extern "C" bsr_status bsr_screened_spmm(const void* A, const float* diag, const void* B, int32_t dtype, int32_t n,
                                        int32_t n_cols, float threshold, void* C, void* stream) {
  if (dtype != BSR_BF16 && dtype != BSR_F16)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_screened_spmm: dtype %d not supported (BSR_BF16 or BSR_F16)", dtype);
  if (n < 1 || n_cols < 1) return fail(BSR_ERR_INVALID_ARG, "bsr_screened_spmm: sizes n %d, n_cols %d", n, n_cols);
  if (n % 128 != 0 || n > 65536)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_screened_spmm: n %d is not a multiple of 128 up to 65536", n);
  if (n_cols % 64 != 0)
    return fail(BSR_ERR_UNSUPPORTED, "bsr_screened_spmm: n_cols %d is not a multiple of 64", n_cols);
  if (!(threshold >= 0.f) || isinf(threshold))
    return fail(BSR_ERR_INVALID_ARG, "bsr_screened_spmm: threshold must be finite and >= 0");
  if (!A || !diag || !B || !C) return fail(BSR_ERR_INVALID_ARG, "bsr_screened_spmm: null pointer");
  if ((((uintptr_t)A) | ((uintptr_t)diag) | ((uintptr_t)B) | ((uintptr_t)C)) & 15)
    return fail(BSR_ERR_INVALID_ARG, "bsr_screened_spmm: data pointer is not 16-byte aligned");
  ScreenedArgs a{A, diag, B, C, n, n_cols, threshold, dtype, status_ptr()};
  if (!a.status) return fail(BSR_ERR_CUDA, "bsr_screened_spmm: no CUDA device");
  return launch_screened_tc(a, (cudaStream_t)stream);
}

extern "C" bsr_status bsr_attn_fwd_two_pass(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                                            const int32_t* row_ptr, const int32_t* col_idx, int32_t n_brows,
                                            int32_t block, float scale, bsr_tensor* O, float* row_max,
                                            float* row_denom, void* stream) {
  return bsr::fwd_impl(Q, K, V, row_ptr, col_idx, n_brows, block, scale, O, row_max, row_denom, stream, true);
}

namespace bsr {

bsr_status build_bwd_args(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const bsr_tensor* O,
                          const bsr_tensor* dO, const float* row_max, const float* row_denom,
                          const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
                          const int32_t* row_idx, float scale, bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV,
                          BwdArgs* out) {
  bsr_status st;
  if ((st = check_tensor(Q, "Q", nullptr)) || (st = check_tensor(K, "K", Q)) || (st = check_tensor(V, "V", Q)) ||
      (st = check_tensor(O, "O", Q)) || (st = check_tensor(dO, "dO", Q)) || (st = check_tensor(dQ, "dQ", Q)) ||
      (st = check_tensor(dK, "dK", Q)) || (st = check_tensor(dV, "dV", Q)))
    return st;
  if (!row_max || !row_denom || !row_ptr || !col_idx || !col_ptr || !row_idx)
    return fail(BSR_ERR_INVALID_ARG, "bsr_attn_bwd: null statistics or structure array");
  BwdArgs a{};
  if ((st = make_dims(Q, scale, &a.d))) return st;
  a.Q = Q->data;
  a.K = K->data;
  a.V = V->data;
  a.O = O->data;
  a.dO = dO->data;
  a.row_max = row_max;
  a.row_denom = row_denom;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.col_ptr = col_ptr;
  a.row_idx = row_idx;
  a.dQ = dQ->data;
  a.dK = dK->data;
  a.dV = dV->data;
  a.status = status_ptr();
  if (!a.status) return fail(BSR_ERR_CUDA, "bsr_attn_bwd: no CUDA device");
  *out = a;
  return BSR_OK;
}

size_t bwd_scratch_bytes(const Dims& d, int G, bool split) {
  const size_t rows = (size_t)d.BH * d.S;
  const int heads = plan_heads(d);
  size_t bytes = 2 * sizeof(float) * rows;
  bytes += 3 * sizeof(int32_t) * plan_words(d.nb, G, heads);
  if (split) bytes += 3 * part_tile_bytes(d, false) * plan_tiles(d.nb, G, heads);
  if (!tc_bwd_supported(d)) bytes += wide_piece_bytes(d, 4);
  return bytes;
}

void bwd_scratch_carve(BwdArgs* a, void* base, int G, bool split) {
  const size_t rows = (size_t)a->d.BH * a->d.S;
  const int heads = plan_heads(a->d);
  const size_t pw = plan_words(a->d.nb, G, heads);
  a->delta = (float*)base;
  a->lse2 = a->delta + rows;
  a->row_plan = (int32_t*)(a->lse2 + rows);
  a->col_plan = a->row_plan + pw;
  a->col_plan2 = a->col_plan + pw;
  char* next = (char*)(a->col_plan2 + pw);
  // partial tiles: one set for dQ, then two for dK / dV
  const size_t set = part_tile_bytes(a->d, false) * plan_tiles(a->d.nb, G, heads);
  a->part_q = split ? (float*)next : nullptr;
  a->part_kv = split ? (float*)(next + set) : nullptr;
  if (split) next += 3 * set;
  a->pieces = tc_bwd_supported(a->d) ? nullptr : (void*)next;
}

bsr_status run_bwd(const BwdArgs& a, cudaStream_t s, bool split, bool planned, bool zero) {
  bsr_status st;
  ZeroArgs z{};
  if (zero) {  // dQ of empty block rows, dK / dV of empty block columns
    z.t[0] = ZeroTarget{a.row_ptr, {a.dQ, nullptr}, nullptr, nullptr};
    z.t[1] = ZeroTarget{a.col_ptr, {a.dK, a.dV}, nullptr, nullptr};
    z.targets = 2;
    z.nb = a.d.nb;
    z.BH = a.d.BH;
    z.S = a.d.S;
    z.row_bytes = a.d.D * (a.d.dtype == BSR_F32 ? 4 : 2);
    // on a plan the zero pass has a launch of its own; otherwise it rides in
    // the planner's launch
    if (planned && (st = launch_zero_lines(z, s)) != BSR_OK) return st;
  }
  if (planned) {  // the work lists are built already (a bsr_plan): delta, then the walks
    if (!tc_bwd_supported(a.d) && !wide_supported(a.d))
      return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_bwd: dtype %d with head_dim %d", a.d.dtype, a.d.D);
    if ((st = launch_delta(a, s)) != BSR_OK) return st;
    return tc_bwd_supported(a.d) ? launch_bwd_tc(a, s) : launch_bwd_wide(a, s);
  }
  PlanArgs p{};
  p.list[0] = PlanList{a.row_ptr, a.row_plan};
  p.list[1] = PlanList{a.col_ptr, a.col_plan};
  p.list[2] = PlanList{a.col_ptr, a.col_plan2};
  p.n = a.d.nb;
  p.G = tc_grid(a.d);
  p.BH = plan_heads(a.d);
  p.allow_split = split ? 1 : 0;
  p.skip_empty = 1;
  p.status = a.status;
  if (zero) {
    p.zero = z;
    p.zero_ctas = zero_ctas(z);
  }
  if (tc_bwd_supported(a.d)) {
    if ((st = launch_delta_plan(a, p, 2, s)) != BSR_OK) return st;
    return launch_bwd_tc(a, s);
  }
  if (!wide_supported(a.d))
    return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_bwd: dtype %d with head_dim %d", a.d.dtype, a.d.D);
  // dQ, dV and dK each on a plan of its own
  if ((st = launch_delta_plan(a, p, 3, s)) != BSR_OK) return st;
  return launch_bwd_wide(a, s);
}

}  // namespace bsr

extern "C" bsr_status bsr_attn_bwd(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
                                   const bsr_tensor* O, const bsr_tensor* dO,
                                   const float* row_max, const float* row_denom,
                                   const int32_t* row_ptr, const int32_t* col_idx,
                                   const int32_t* col_ptr, const int32_t* row_idx,
                                   float scale,
                                   bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV, void* stream) {
  BwdArgs a{};
  bsr_status st = build_bwd_args(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale,
                                 dQ, dK, dV, &a);
  if (st != BSR_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int G = tc_grid(a.d);
  if (G <= 0) return fail(BSR_ERR_CUDA, "bsr_attn_bwd: cannot query the SM count");
  const size_t scratch_bytes = bwd_scratch_bytes(a.d, G, true);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, scratch_bytes, s);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "bsr_attn_bwd: cudaMallocAsync(%zu): %s", scratch_bytes, cudaGetErrorString(e));
  bwd_scratch_carve(&a, scratch, G, true);
  st = run_bwd(a, s, true, false, true);
  e = cudaFreeAsync(scratch, s);
  if (st == BSR_OK && e != cudaSuccess) st = fail(BSR_ERR_CUDA, "bsr_attn_bwd: cudaFreeAsync: %s", cudaGetErrorString(e));
  return st;
}

extern "C" bsr_status bsr_attn_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_attn_check: %s", cudaGetErrorString(e));
  int* p = status_ptr();
  if (!p) return fail(BSR_ERR_CUDA, "bsr_attn_check: no CUDA device");
  int v = 0, zero = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_attn_check: %s", cudaGetErrorString(e));
  if (v == kStatusTimeout) return fail(BSR_ERR_TIMEOUT, "a bounded device-side wait gave up");
  if (v == kStatusDeviceCheck) return fail(BSR_ERR_DEVICE_CHECK, "a device-side index check failed (block index out of range)");
  if (v != 0) return fail(BSR_ERR_CUDA, "unknown device status %d", v);
  return BSR_OK;
}

extern "C" bsr_status bsr_set_wait_limit(uint64_t ns) {
  int* p = status_ptr();
  if (!p) return fail(BSR_ERR_CUDA, "bsr_set_wait_limit: no CUDA device");
  const unsigned long long v = ns ? (unsigned long long)ns : kDefaultWaitLimitNs;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(p + 2, &v, sizeof(v), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_set_wait_limit: %s", cudaGetErrorString(e));
  return BSR_OK;
}

extern "C" void bsr_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
}

extern "C" int32_t bsr_profile_collect(bsr_kernel_time* out, int32_t max_entries) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  std::vector<bsr_kernel_time> agg;
  for (auto& t : g_prof) {
    float ms = 0.f;
    cudaEventSynchronize(t.stop);
    cudaEventElapsedTime(&ms, t.start, t.stop);
    size_t k = 0;
    for (; k < agg.size(); ++k)
      if (t.name == agg[k].name) break;
    if (k == agg.size()) {
      bsr_kernel_time z{};
      strncpy(z.name, t.name.c_str(), sizeof(z.name) - 1);
      agg.push_back(z);
    }
    agg[k].launches += 1;
    agg[k].total_ms += ms;
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_prof.clear();
  int32_t n = 0;
  for (auto& a : agg) {
    if (n >= max_entries) break;
    if (out) out[n] = a;
    ++n;
  }
  return n;
}
