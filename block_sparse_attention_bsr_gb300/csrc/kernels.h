// Kernel-side declarations: argument blocks and launchers for the attention
// kernels.  Shared by the C-ABI front end and the kernel translation units.
#pragma once

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
  const int32_t* order;  // [nb] block rows longest first (plan_kernel), or null
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
  int32_t* row_order;  // [nb] scratch: block rows longest first
  int32_t* col_order;  // [nb] scratch: block columns longest first
  int* status;
};

// Planner inputs: one or two prefix-offset lists of n lines each.
struct PlanArgs {
  const int32_t* ptr0;
  const int32_t* ptr1;
  int32_t* order0;
  int32_t* order1;
  int n;
};

// Sorts the lines of `lists` (1 or 2) prefix-offset lists by length, longest
// first, into the order arrays.
bsr_status launch_plan(const PlanArgs& p, int lists, cudaStream_t s);

// RAII bracket that records a pair of CUDA events around one kernel launch
// when profiling is enabled (bsr_profile_enable).
class LaunchTimer {
 public:
  LaunchTimer(const char* name, cudaStream_t stream);
  ~LaunchTimer();

 private:
  int slot_;
  cudaStream_t stream_;
};

// Validates the backward arguments and fills *out (delta left null).
bsr_status build_bwd_args(const bsr_tensor* Q, const bsr_tensor* K, const bsr_tensor* V, const bsr_tensor* O,
                          const bsr_tensor* dO, const float* row_max, const float* row_denom,
                          const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
                          const int32_t* row_idx, float scale, bsr_tensor* dQ, bsr_tensor* dK, bsr_tensor* dV,
                          BwdArgs* out);

// Launches the backward kernels (plan, delta, dQ, dK/dV) on `s`; a.delta and
// a.lse2 must each point at BH * S floats of 16-byte aligned device scratch,
// a.row_order and a.col_order at nb ints each.
bsr_status run_bwd(const BwdArgs& a, cudaStream_t s);

// Returns a status for the last launch on this thread (cudaGetLastError).
bsr_status check_launch(const char* what);

// Portable SIMT kernels (every head_dim and dtype).
bsr_status launch_fwd_simt(const FwdArgs& a, cudaStream_t s);
bsr_status launch_delta(const BwdArgs& a, cudaStream_t s);
bsr_status launch_dq_simt(const BwdArgs& a, cudaStream_t s);
bsr_status launch_dkdv_simt(const BwdArgs& a, cudaStream_t s);

// Tensor-core (tcgen05 / TMA) kernels.  `order` (device, optional) maps the
// CTA's x index to a block row.
bool tc_fwd_supported(const Dims& d);
bsr_status launch_fwd_tc(const FwdArgs& a, const int32_t* order, cudaStream_t s);
bsr_status launch_fwd_tc2(const FwdArgs& a, cudaStream_t s);  // head_dim 64 / 128, P in TMEM
bool tc_bwd_supported(const Dims& d);
bsr_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s);

}  // namespace bsr
