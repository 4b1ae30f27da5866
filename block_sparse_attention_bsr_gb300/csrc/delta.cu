// The delta pass of the backward: D_i = dO_i . O_i and the base-2
// log-sum-exp lse2_i = row_max_i log2(e) + log2(row_denom_i), one fp32 value
// each per query row ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.5.0]:
// the delta identity).  An HBM-bound elementwise pass over O and dO (no
// contraction), for every operand type and head_dim; the 16-bit head_dim
// 64 / 128 backward runs the same rows fused with its planner (plan.cu).

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "delta.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace bsr {
namespace {

constexpr int kThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) delta_kernel(BwdArgs a) {
  sm100::griddep_wait();  // may run as a programmatic dependent of the forward
  sm100::griddep_launch_dependents();
  delta_pass<T, D, kThreads>(a, blockIdx.x, gridDim.x);
}

template <typename T, int D>
bsr_status delta_dispatch(const BwdArgs& a, cudaStream_t s) {
  const size_t rows = (size_t)a.d.BH * a.d.S;
  constexpr size_t per = delta_rows_per_cta<T, D, kThreads>();
  const size_t groups = (rows + per - 1) / per;
  const dim3 grid((unsigned)groups);  // one CTA per row group (DeltaShape)
  LaunchTimer timer("delta", s);
  const cudaError_t e = launch_dependent(delta_kernel<T, D>, grid, dim3(kThreads), 0, s, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "delta launch: %s", cudaGetErrorString(e));
  return check_launch("delta launch");
}

template <typename T>
bsr_status delta_dim(const BwdArgs& a, cudaStream_t s) {
  switch (a.d.D) {
    case 64: return delta_dispatch<T, 64>(a, s);
    case 128: return delta_dispatch<T, 128>(a, s);
    case 256: return delta_dispatch<T, 256>(a, s);
    case 512: return delta_dispatch<T, 512>(a, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "delta: head_dim %d not supported", a.d.D);
  }
}

// Outputs of empty lines on their own launch (zero_lines_body, delta.cuh);
// the per-call entry points run the same body in extra CTAs of their
// planner launch instead.
__global__ void __launch_bounds__(kThreads) zero_lines_kernel(ZeroArgs z) {
  sm100::griddep_wait();  // may run as a programmatic dependent
  sm100::griddep_launch_dependents();
  zero_lines_body(z, blockIdx.x, gridDim.x);
}

}  // namespace

bsr_status launch_zero_lines(const ZeroArgs& z, cudaStream_t s) {
  if (z.targets < 1 || z.targets > 2 || z.row_bytes % 16 != 0)
    return fail(BSR_ERR_INVALID_ARG, "zero_lines: %d targets, %d-byte rows", z.targets, z.row_bytes);
  const long long pairs = (long long)z.nb * z.BH * z.targets;
  const int sms = sm_count();
  const long long cap = sms > 0 ? 4LL * sms : 1;
  const dim3 grid((unsigned)(pairs < cap ? (pairs > 0 ? pairs : 1) : cap));
  LaunchTimer timer("zero_lines", s);
  const cudaError_t e = launch_dependent(zero_lines_kernel, grid, dim3(kThreads), 0, s, z);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "zero_lines launch: %s", cudaGetErrorString(e));
  return check_launch("zero_lines launch");
}

bsr_status launch_delta(const BwdArgs& a, cudaStream_t s) {
  if (a.d.dtype == BSR_BF16) return delta_dim<__nv_bfloat16>(a, s);
  if (a.d.dtype == BSR_F16) return delta_dim<__half>(a, s);
  return delta_dim<float>(a, s);
}

}  // namespace bsr
