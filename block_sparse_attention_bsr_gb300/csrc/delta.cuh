// Per-query-row statistics of the backward pass, shared by the standalone
// delta kernel and the fused delta + planner kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stddef.h>

#include "kernels.h"

namespace bsr {

// D_i = dO_i . O_i (fp32) and the base-2 log-sum-exp of the row,
// lse2_i = row_max_i log2(e) + log2(row_denom_i), one value each per query
// row.  G lanes share a row, each reading 8 contiguous elements per step.

// 8 contiguous elements in registers, as loaded.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
};
template <>
struct Raw8<__half> {
  uint4 v;
};
template <>
struct Raw8<float> {
  float4 v0, v1;
};

__device__ __forceinline__ Raw8<__nv_bfloat16> ld8(const __nv_bfloat16* p) { return Raw8<__nv_bfloat16>{*(const uint4*)p}; }
__device__ __forceinline__ Raw8<__half> ld8(const __half* p) { return Raw8<__half>{*(const uint4*)p}; }
__device__ __forceinline__ Raw8<float> ld8(const float* p) {
  return Raw8<float>{*(const float4*)p, *(const float4*)(p + 4)};
}

__device__ __forceinline__ float dot8(const Raw8<__nv_bfloat16>& a, const Raw8<__nv_bfloat16>& b) {
  const __nv_bfloat162* xa = (const __nv_bfloat162*)&a.v;
  const __nv_bfloat162* ya = (const __nv_bfloat162*)&b.v;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __bfloat1622float2(xa[k]), v = __bfloat1622float2(ya[k]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}
__device__ __forceinline__ float dot8(const Raw8<__half>& a, const Raw8<__half>& b) {
  const __half2* xa = (const __half2*)&a.v;
  const __half2* ya = (const __half2*)&b.v;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __half22float2(xa[k]), v = __half22float2(ya[k]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}
__device__ __forceinline__ float dot8(const Raw8<float>& a, const Raw8<float>& b) {
  float s = a.v0.x * b.v0.x;
  s = fmaf(a.v0.y, b.v0.y, s);
  s = fmaf(a.v0.z, b.v0.z, s);
  s = fmaf(a.v0.w, b.v0.w, s);
  s = fmaf(a.v1.x, b.v1.x, s);
  s = fmaf(a.v1.y, b.v1.y, s);
  s = fmaf(a.v1.z, b.v1.z, s);
  s = fmaf(a.v1.w, b.v1.w, s);
  return s;
}

// Lanes per row, 8-element chunks per lane and row, and rows per lane group
// handled in one pass: all of a pass's loads are issued before any of them
// is used (about 64 bytes of operands per lane, fewer rows when the rows
// are wide).  The groups are small and every group gets a CTA of its own,
// so that the CTAs fill each SM as soon as the forward's CTAs leave it;
// four times the rows per group, looped over by as many CTAs as the SMs
// hold at once, made the step ~4 µs slower at seq 8192.
template <typename T, int D>
struct DeltaShape {
  static constexpr int CH = D / 8;              // 8-element chunks per row
  static constexpr int G = CH < 32 ? CH : 32;   // lanes per row
  static constexpr int NCH = CH / G;            // chunks per lane and row
  static constexpr int RPW = 32 / G;            // rows per warp and pass step
  static constexpr int kBytes = 2 * NCH * 8 * (int)sizeof(T);  // per lane and row
  static constexpr int U = kBytes <= 64 ? 2 : 1;
};

template <typename T, int D, int kThreads>
__host__ __device__ constexpr int delta_rows_per_cta() {
  return (kThreads / 32) * DeltaShape<T, D>::RPW * DeltaShape<T, D>::U;
}

// The rows of CTA `cta` (kThreads threads) of a delta pass.  Row indices
// past the end are clamped for the loads (so no load sits under a branch
// and all of them are in flight together) and their results dropped.
template <typename T, int D, int kThreads>
__device__ __forceinline__ void delta_rows(const BwdArgs& a, int cta) {
  using Sh = DeltaShape<T, D>;
  constexpr int G = Sh::G, NCH = Sh::NCH, RPW = Sh::RPW, U = Sh::U;
  static_assert(Sh::CH % G == 0, "whole chunks per lane");
  constexpr int kPer = delta_rows_per_cta<T, D, kThreads>();
  static_assert(128 % kPer == 0, "a group of rows lies inside one block row");
  // The rows of a block row with no stored block are in no work item, and
  // no kernel reads their statistics: the group skips them.
  {
    const int m = (int)(((size_t)cta * kPer % (size_t)a.d.S) / 128);
    if (a.row_ptr[m + 1] == a.row_ptr[m]) return;
  }
  const int lane = threadIdx.x % 32;
  const size_t rows = (size_t)a.d.BH * a.d.S;
  const size_t row0 = ((size_t)cta * (kThreads / 32) + threadIdx.x / 32) * RPW * U + lane / G;
  Raw8<T> ov[U][NCH], gv[U][NCH];
  float rmax[U], rden[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const size_t row = row0 + (size_t)u * RPW;
    const size_t rr = row < rows ? row : rows - 1;
    const T* o = (const T*)a.O + rr * D;
    const T* g = (const T*)a.dO + rr * D;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = lane % G + k * G;
      ov[u][k] = ld8(o + c * 8);
      gv[u][k] = ld8(g + c * 8);
    }
    rmax[u] = a.row_max[rr];
    rden[u] = a.row_denom[rr];
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; ++k) t += dot8(ov[u][k], gv[u][k]);
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const size_t row = row0 + (size_t)u * RPW;
    if (row < rows && lane % G == 0) {
      a.delta[row] = t;
      a.lse2[row] = rmax[u] * 1.4426950408889634f + log2f(rden[u]);
    }
  }
}

// A whole delta pass over the rows, in groups of delta_rows_per_cta rows:
// CTA `first` of `stride` takes groups first, first + stride, ... (the
// launches give every group a CTA, so each takes one).
template <typename T, int D, int kThreads>
__device__ __forceinline__ void delta_pass(const BwdArgs& a, int first, int stride) {
  const size_t rows = (size_t)a.d.BH * a.d.S;
  constexpr size_t per = delta_rows_per_cta<T, D, kThreads>();
  const int groups = (int)((rows + per - 1) / per);
  for (int c = first; c < groups; c += stride) delta_rows<T, D, kThreads>(a, c);
}

// Outputs of empty lines (no stored block): the work lists leave those
// lines out (PlanArgs::skip_empty), so no attention kernel visits them; this
// writes what the method gives them instead: zero output rows, and for the
// forward row_max = -inf, row_denom = 0 (no key is attended).  CTA `cta` of
// `ncta` takes the (target, line, head) triples cta, cta + ncta, ...; a line
// is empty when its two offsets agree.  Needs blockDim.x >= 128.
__device__ __forceinline__ void zero_lines_body(const ZeroArgs& z, int cta, int ncta) {
  const long long per = (long long)z.nb * z.BH;
  for (long long w = cta; w < per * z.targets; w += ncta) {
    const ZeroTarget& t = w >= per ? z.t[1] : z.t[0];
    const int line = (int)(w % per % z.nb), bh = (int)(w % per / z.nb);
    if (t.ptr[line + 1] != t.ptr[line]) continue;
    const size_t row0 = (size_t)bh * z.S + (size_t)line * 128;
    const size_t n16 = (size_t)128 * z.row_bytes / 16;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int k = 0; k < 2; ++k) {
      if (!t.out[k]) continue;
      uint4* o = (uint4*)((char*)t.out[k] + row0 * z.row_bytes);
      for (size_t i = threadIdx.x; i < n16; i += blockDim.x) o[i] = zero;
    }
    if (t.row_max && threadIdx.x < 128) {
      t.row_max[row0 + threadIdx.x] = -INFINITY;
      t.row_denom[row0 + threadIdx.x] = 0.f;
    }
  }
}

}  // namespace bsr
