// Work ordering for the attention kernels: block rows (or block columns)
// sorted by their number of stored blocks, longest first.
//
// The pages split output tiles between cores "balanced by stored blocks"
// with one writer per tile ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG
// [0.9.0]).  Here the same balance comes from the launch order: the CTA with
// linear index c handles line order[c / BH] of head c % BH, so the longest
// lines of every head start in the first wave and the short ones fill in
// behind them.  Each output tile is still written by exactly one CTA.
//
// One CTA per list: a counting sort by count (descending).  Lines with the
// same count may come out in any order; that changes only the schedule, never
// a result.

#include "kernels.h"

namespace bsr {
namespace {

constexpr int kPlanThreads = 1024;

// ptr: [n + 1] prefix offsets; order: [n] out.  hist: n + 1 ints of shared memory.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs p) {
  extern __shared__ int hist[];
  const int* ptr = blockIdx.x == 0 ? p.ptr0 : p.ptr1;
  int* order = blockIdx.x == 0 ? p.order0 : p.order1;
  const int n = p.n;
  for (int v = threadIdx.x; v <= n; v += blockDim.x) hist[v] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int c = ptr[i + 1] - ptr[i];
    c = c < 0 ? 0 : (c > n ? n : c);
    atomicAdd(&hist[c], 1);
  }
  __syncthreads();
  // exclusive scan from the largest count down: start[v] = #lines with count > v
  if (threadIdx.x == 0) {
    int run = 0;
    for (int v = n; v >= 0; --v) {
      const int h = hist[v];
      hist[v] = run;
      run += h;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int c = ptr[i + 1] - ptr[i];
    c = c < 0 ? 0 : (c > n ? n : c);
    order[atomicAdd(&hist[c], 1)] = i;
  }
}

}  // namespace

bsr_status launch_plan(const PlanArgs& p, int lists, cudaStream_t s) {
  const size_t smem = sizeof(int) * (size_t)(p.n + 1);
  if (smem > 200 * 1024) return fail(BSR_ERR_UNSUPPORTED, "plan: %d block rows exceed the planner's limit", p.n);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "plan: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  LaunchTimer timer("plan", s);
  plan_kernel<<<lists, kPlanThreads, smem, s>>>(p);
  return check_launch("plan launch");
}

}  // namespace bsr
