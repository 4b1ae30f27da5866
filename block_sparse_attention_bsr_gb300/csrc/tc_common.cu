// TMA tensor-map encoding through the driver entry point (no link-time
// dependency on libcuda).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tc_common.h"

namespace bsr {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}
}  // namespace

bsr_status make_tensor_map(const Dims& d, const void* ptr, CUtensorMap* map, const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(BSR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (((uintptr_t)ptr) & 15) return fail(BSR_ERR_INVALID_ARG, "%s: data pointer is not 16-byte aligned", what);
  const cuuint32_t elem = d.dtype == BSR_F32 ? 4 : 2;
  const CUtensorMapDataType type = d.dtype == BSR_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : d.dtype == BSR_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t dims[2] = {(cuuint64_t)d.D, (cuuint64_t)d.BH * (cuuint64_t)d.S};
  const cuuint64_t strides[1] = {(cuuint64_t)d.D * elem};
  const cuuint32_t box[2] = {128 / elem, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, type, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(BSR_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
  return BSR_OK;
}

bsr_status make_tensor_maps(const Dims& d, const void* Q, const void* K, const void* V, TensorMaps* out) {
  bsr_status st;
  if (Q && (st = make_tensor_map(d, Q, &out->q, "Q"))) return st;
  if (K && (st = make_tensor_map(d, K, &out->k, "K"))) return st;
  if (V && (st = make_tensor_map(d, V, &out->v, "V"))) return st;
  return BSR_OK;
}

}  // namespace bsr
