// Host-side helpers shared by the tensor-core kernels: TMA tensor maps over
// the [batch * heads * seq, head_dim] row-major operands.
#pragma once

#include <cuda.h>

#include "kernels.h"

namespace bsr {

struct TensorMaps {
  CUtensorMap q, k, v;
};

// Encodes 2-D tensor maps (inner dimension = head_dim, outer = batch * heads *
// seq rows) with 128-row x 128-byte boxes and the 128-byte swizzle for
// Q, K and V (any of them may be null and is then skipped).
bsr_status make_tensor_maps(const Dims& d, const void* Q, const void* K, const void* V, TensorMaps* out);

// Encodes one such map for `ptr` into *map.
bsr_status make_tensor_map(const Dims& d, const void* ptr, CUtensorMap* map, const char* what);

}  // namespace bsr
