// Backward pass that allocates nothing, for callers that cannot allocate
// device memory.
//
// bsr_attn_bwd takes its scratch (two fp32 values per query row: the delta
// D_i = dO_i . O_i and the row's base-2 log-sum-exp) from cudaMallocAsync
// on the caller's stream.  Some callers cannot allow that: their device memory is
// already fully reserved by another allocator (a framework's caching
// allocator that holds the whole device, or a serving runtime that carves
// all memory into its own pools), or their hot path is not allowed to call
// into the CUDA allocator at all.  bsr_attn_bwd_noalloc runs the same
// kernels but takes that scratch from a fixed-size array in the library's
// static device memory instead.
//
// Limits and rules:
//  * The array holds 2 * kNoAllocMaxRows floats plus kNoAllocPlanWords ints
//    for the work lists (9 MiB in all), so batch * heads * seq must not
//    exceed 1,048,576 (e.g. 128 heads at seq 8192).  fp32 operands also keep
//    their bf16 pieces there (3 pieces of Q, K, V and dO: 24 bytes per
//    element of Q), which caps fp32 calls near batch * heads * seq *
//    head_dim = 390,000.  Larger calls are rejected with
//    BSR_ERR_INVALID_ARG.  Every GPU that loads the library keeps the array
//    reserved until the process exits.
//  * Long block rows / columns are not split into chunks here (that needs
//    partial-result buffers); the work is still spread longest first.
//  * All calls share the one array.  The delta kernel overwrites every entry
//    that is later read, so nothing has to start at zero, but two calls whose
//    kernels overlap on the GPU (different streams, or different host
//    threads on the same device) race on the array: order them.
//  * The device address of the array is looked up once per device, on the
//    first call made with that device current; make that first call before
//    any stream capture.  The address is kept for the life of the process:
//    do not call this entry point after cudaDeviceReset, which destroys the
//    primary context that the address belongs to.

#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace bsr {
namespace {

constexpr size_t kNoAllocMaxRows = size_t(1) << 20;

constexpr size_t kNoAllocPlanWords = size_t(1) << 18;

static __device__ __align__(256) float g_noalloc_delta[2 * kNoAllocMaxRows + kNoAllocPlanWords];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_delta on the current device (host code must not
// use the symbol itself: on the host it names a stand-in, not device memory).
bsr_status noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "bsr_attn_bwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(BSR_ERR_UNSUPPORTED, "bsr_attn_bwd_noalloc: device %d", dev);
  static std::mutex mu;
  static float* cache[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    float* ptr = nullptr;
    e = cudaGetSymbolAddress((void**)&ptr, g_noalloc_delta);
    if (e != cudaSuccess || !ptr)
      return fail(BSR_ERR_CUDA, "bsr_attn_bwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    cache[dev] = ptr;
  }
  *out = cache[dev];
  return BSR_OK;
}

}  // namespace
}  // namespace bsr

using namespace bsr;

extern "C" bsr_status bsr_attn_bwd_noalloc(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V,
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
  const size_t rows = (size_t)a.d.BH * (size_t)a.d.S;
  if (rows > kNoAllocMaxRows)
    return fail(BSR_ERR_INVALID_ARG,
                "bsr_attn_bwd_noalloc: batch * heads * seq = %zu exceeds the static scratch of %zu rows; "
                "use bsr_attn_bwd",
                rows, kNoAllocMaxRows);
  const int G = tc_grid(a.d);
  if (G <= 0) return fail(BSR_ERR_CUDA, "bsr_attn_bwd_noalloc: cannot query the SM count");
  if (bwd_scratch_bytes(a.d, G, false) > sizeof(g_noalloc_delta))
    return fail(BSR_ERR_INVALID_ARG,
                "bsr_attn_bwd_noalloc: the work lists (and, for fp32 operands, their bf16 pieces) need more than "
                "the static scratch of %zu bytes; use bsr_attn_bwd",
                sizeof(g_noalloc_delta));
  float* base = nullptr;
  if ((st = noalloc_scratch(&base)) != BSR_OK) return st;
  bwd_scratch_carve(&a, base, G, false);
  return run_bwd(a, (cudaStream_t)stream, false, false, true);
}
