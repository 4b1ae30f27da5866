// Per-query-row statistics of the backward pass, shared by the standalone
// delta kernel and the fused delta + planner kernel.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stddef.h>

#include "kernels.h"

namespace bsr {

// D_i = dO_i . O_i (fp32) and the base-2 log-sum-exp of the row,
// lse2_i = row_max_i log2(e) + log2(row_denom_i), one value each per query
// row.  G lanes share a row, each reading 8 contiguous elements per step.
template <typename T>
__device__ __forceinline__ float dot8(const T* a, const T* b);
template <>
__device__ __forceinline__ float dot8<__nv_bfloat16>(const __nv_bfloat16* a, const __nv_bfloat16* b) {
  const uint4 x = *(const uint4*)a, y = *(const uint4*)b;
  const __nv_bfloat162* xa = (const __nv_bfloat162*)&x;
  const __nv_bfloat162* ya = (const __nv_bfloat162*)&y;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __bfloat1622float2(xa[k]), v = __bfloat1622float2(ya[k]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}
template <>
__device__ __forceinline__ float dot8<float>(const float* a, const float* b) {
  const float4 x0 = *(const float4*)a, x1 = *(const float4*)(a + 4);
  const float4 y0 = *(const float4*)b, y1 = *(const float4*)(b + 4);
  float s = x0.x * y0.x;
  s = fmaf(x0.y, y0.y, s);
  s = fmaf(x0.z, y0.z, s);
  s = fmaf(x0.w, y0.w, s);
  s = fmaf(x1.x, y1.x, s);
  s = fmaf(x1.y, y1.y, s);
  s = fmaf(x1.z, y1.z, s);
  s = fmaf(x1.w, y1.w, s);
  return s;
}

// Rows handled by one lane group in one pass: all their loads are issued
// before any reduction, so enough bytes are in flight to keep HBM busy.
constexpr int kDeltaUnroll = 4;

template <int D, int kThreads>
__host__ __device__ constexpr int delta_rows_per_cta() {
  return (kThreads / 32) * (32 / (D / 8 < 32 ? D / 8 : 32)) * kDeltaUnroll;
}

// The rows of CTA `cta` (kThreads threads) of a delta pass.
template <typename T, int D, int kThreads>
__device__ __forceinline__ void delta_rows(const BwdArgs& a, int cta) {
  constexpr int CH = D / 8;              // 8-element chunks per row
  constexpr int G = CH < 32 ? CH : 32;   // lanes per row
  constexpr int RPW = 32 / G;            // rows per warp and unroll step
  constexpr int U = kDeltaUnroll;
  const int lane = threadIdx.x % 32;
  const size_t rows = (size_t)a.d.BH * a.d.S;
  const size_t row0 = ((size_t)cta * (kThreads / 32) + threadIdx.x / 32) * RPW * U + lane / G;
  // the row statistics are loaded with the operands (one round trip to
  // memory, not two), by the lane that writes the row's results
  float s[U], rmax[U], rden[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    s[u] = 0.f;
    rmax[u] = 0.f;
    rden[u] = 1.f;
    const size_t row = row0 + (size_t)u * RPW;
    if (row < rows) {
      if (lane % G == 0) {
        rmax[u] = a.row_max[row];
        rden[u] = a.row_denom[row];
      }
      const T* o = (const T*)a.O + row * D;
      const T* g = (const T*)a.dO + row * D;
#pragma unroll
      for (int c = lane % G; c < CH; c += G) s[u] += dot8<T>(o + c * 8, g + c * 8);
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float t = s[u];
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const size_t row = row0 + (size_t)u * RPW;
    if (row < rows && lane % G == 0) {
      a.delta[row] = t;
      a.lse2[row] = rmax[u] * 1.4426950408889634f + log2f(rden[u]);
    }
  }
}

}  // namespace bsr
