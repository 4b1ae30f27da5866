// Portable SIMT kernels for block-sparse attention (fp32 arithmetic).
//
// They serve every supported head_dim (64/128/256/512) and every operand type
// (fp32; bf16 and fp16 widened to fp32), with the same walk as the
// tensor-core kernels:
//   * forward: one CTA per 16 query rows of a block row m, walking the row's
//     stored blocks j in [row_ptr[m], row_ptr[m+1]) and the 128 keys of block
//     col_idx[j] in chunks, with an online softmax ("trnsparse 0.7.0 -> 0.9.0"
//     diff, CHANGELOG [0.8.0]: one launch, statistics on chip, K/V addressed
//     by block column with no gather);
//   * delta: D_i = dO_i . O_i ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG
//     [0.5.0], Flash Attention delta identity);
//   * dQ: row-first walk, dQ_m += scale dS K_n ("trnsparse 0.4.1 -> 0.6.0"
//     diff, CHANGELOG [0.5.1], _attn_bwd_dq_kernel);
//   * dK/dV: column-first walk over the BSC lists, dV_n += P^T dO_m,
//     dK_n += scale dS^T Q_m (same CHANGELOG entry, _attn_bwd_dkdv_kernel).
// Every output element has exactly one writer; no atomics touch outputs.

#include <cuda_bf16.h>
#include <math.h>

#include "delta.cuh"
#include "kernels.h"

namespace bsr {
namespace {

constexpr int kRowsPerCta = 16;  // query (or key) rows per CTA
constexpr int kThreads = 256;
constexpr int kBlock = 128;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// Copies `rows` contiguous rows of D elements into fp32 shared memory with row stride `ld`.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src, int rows) {
  for (int e = threadIdx.x; e < rows * D; e += blockDim.x) {
    const int r = e / D, c = e % D;
    dst[r * ld + c] = to_f(src[(size_t)r * D + c]);
  }
}

// Reductions across the `W` lanes (a power of two <= 32) that share a row.
template <int W>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int D>
__device__ __forceinline__ float dot(const float* a, const float* b) {
  float s = 0.f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) s = fmaf(a[d], b[d], s);
  return s;
}

__device__ __forceinline__ bool bad_block(int n, int nb, int* status) {
  if (n < 0 || n >= nb) {
    atomicExch(status, kStatusDeviceCheck);
    return true;
  }
  return false;
}

// ---------------------------------------------------------------- forward --
// Warp w owns rows 2w, 2w+1 of the CTA's 16 for the score / softmax phase;
// each lane holds PER = 2*KC/32 scores.  For the P.V phase thread t owns row
// t/16 and columns t%16 + 16 i of the output.
template <typename T, int D, int KC>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
  constexpr int QR = kRowsPerCta;
  constexpr int PER = 2 * KC / 32;
  constexpr int NO = D / 16;
  extern __shared__ float sm[];
  float* Qs = sm;                  // [QR][D]
  float* Ks = Qs + QR * D;         // [KC][D+1]
  float* Vs = Ks + KC * (D + 1);   // [KC][D]
  float* Ps = Vs + KC * D;         // [QR][KC]
  float* alpha_s = Ps + QR * KC;   // [QR]
  float* m_s = alpha_s + QR;       // [QR]
  float* l_s = m_s + QR;           // [QR]

  const int subs = kBlock / QR;
  const int m = blockIdx.x / subs;
  const int q0 = m * kBlock + (blockIdx.x % subs) * QR;
  const int bh = blockIdx.y;
  const size_t head = (size_t)bh * a.d.S * D;
  const T* Q = (const T*)a.Q + head;
  const T* K = (const T*)a.K + head;
  const T* V = (const T*)a.V + head;
  const float scale = a.d.scale;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int orow = threadIdx.x / 16, ocol = threadIdx.x % 16;

  load_rows<T, D>(Qs, D, Q + (size_t)q0 * D, QR);

  float m_run[PER], l_run[PER], acc[NO];
#pragma unroll
  for (int t = 0; t < PER; ++t) { m_run[t] = -INFINITY; l_run[t] = 0.f; }
#pragma unroll
  for (int i = 0; i < NO; ++i) acc[i] = 0.f;

  const int j0 = a.row_ptr[m], j1 = a.row_ptr[m + 1];
  for (int j = j0; j < j1; ++j) {
    const int n = a.col_idx[j];
    if (bad_block(n, a.d.nb, a.status)) continue;
    for (int kc = 0; kc < kBlock; kc += KC) {
      const int k0 = n * kBlock + kc;
      __syncthreads();
      load_rows<T, D>(Ks, D + 1, K + (size_t)k0 * D, KC);
      load_rows<T, D>(Vs, D, V + (size_t)k0 * D, KC);
      __syncthreads();
#pragma unroll
      for (int t = 0; t < PER; ++t) {
        const int e = lane + 32 * t;
        const int r = 2 * warp + e / KC, key = e % KC;
        const float s = scale * dot<D>(Qs + r * D, Ks + key * (D + 1));
        const float mn = fmaxf(m_run[t], group_max<KC>(s));
        const float alpha = (m_run[t] == -INFINITY) ? 0.f : expf(m_run[t] - mn);
        const float p = expf(s - mn);
        l_run[t] = l_run[t] * alpha + group_sum<KC>(p);
        m_run[t] = mn;
        Ps[r * KC + key] = p;
        if (key == 0) alpha_s[r] = alpha;
      }
      __syncthreads();
      const float al = alpha_s[orow];
#pragma unroll
      for (int i = 0; i < NO; ++i) acc[i] *= al;
      for (int jj = 0; jj < KC; ++jj) {
        const float p = Ps[orow * KC + jj];
        const float* vrow = Vs + jj * D + ocol;
#pragma unroll
        for (int i = 0; i < NO; ++i) acc[i] = fmaf(p, vrow[16 * i], acc[i]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < PER; ++t) {
    const int e = lane + 32 * t;
    if (e % KC == 0) {
      const int r = 2 * warp + e / KC;
      m_s[r] = m_run[t];
      l_s[r] = l_run[t];
    }
  }
  __syncthreads();
  const float l = l_s[orow];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* O = (T*)a.O + head + (size_t)(q0 + orow) * D + ocol;
#pragma unroll
  for (int i = 0; i < NO; ++i) O[16 * i] = from_f<T>(acc[i] * inv);
  if (threadIdx.x < QR) {
    const size_t row = (size_t)bh * a.d.S + q0 + threadIdx.x;
    a.row_max[row] = m_s[threadIdx.x];
    a.row_denom[row] = l_s[threadIdx.x];
  }
}

// ------------------------------------------------------------------ delta --
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) delta_kernel(BwdArgs a) {
  delta_pass<T, D, kThreads>(a, blockIdx.x, gridDim.x);
}

// --------------------------------------------------------------------- dQ --
template <typename T, int D, int KC>
__global__ void __launch_bounds__(kThreads) dq_simt_kernel(BwdArgs a) {
  constexpr int QR = kRowsPerCta;
  constexpr int PER = 2 * KC / 32;
  constexpr int NO = D / 16;
  extern __shared__ float sm[];
  float* Qs = sm;                   // [QR][D]
  float* dOs = Qs + QR * D;         // [QR][D]
  float* Ks = dOs + QR * D;         // [KC][D+1]
  float* Vs = Ks + KC * (D + 1);    // [KC][D+1]
  float* DSs = Vs + KC * (D + 1);   // [QR][KC]

  const int subs = kBlock / QR;
  const int m = blockIdx.x / subs;
  const int q0 = m * kBlock + (blockIdx.x % subs) * QR;
  const int bh = blockIdx.y;
  const size_t head = (size_t)bh * a.d.S * D;
  const T* K = (const T*)a.K + head;
  const T* V = (const T*)a.V + head;
  const float scale = a.d.scale;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int orow = threadIdx.x / 16, ocol = threadIdx.x % 16;

  load_rows<T, D>(Qs, D, (const T*)a.Q + head + (size_t)q0 * D, QR);
  load_rows<T, D>(dOs, D, (const T*)a.dO + head + (size_t)q0 * D, QR);

  float rm[PER], rd[PER], dl[PER], acc[NO];
#pragma unroll
  for (int t = 0; t < PER; ++t) {
    const int r = 2 * warp + (lane + 32 * t) / KC;
    const size_t row = (size_t)bh * a.d.S + q0 + r;
    rm[t] = a.row_max[row];
    rd[t] = a.row_denom[row];
    dl[t] = a.delta[row];
  }
#pragma unroll
  for (int i = 0; i < NO; ++i) acc[i] = 0.f;

  const int j0 = a.row_ptr[m], j1 = a.row_ptr[m + 1];
  for (int j = j0; j < j1; ++j) {
    const int n = a.col_idx[j];
    if (bad_block(n, a.d.nb, a.status)) continue;
    for (int kc = 0; kc < kBlock; kc += KC) {
      const int k0 = n * kBlock + kc;
      __syncthreads();
      load_rows<T, D>(Ks, D + 1, K + (size_t)k0 * D, KC);
      load_rows<T, D>(Vs, D + 1, V + (size_t)k0 * D, KC);
      __syncthreads();
#pragma unroll
      for (int t = 0; t < PER; ++t) {
        const int e = lane + 32 * t;
        const int r = 2 * warp + e / KC, key = e % KC;
        const float s = scale * dot<D>(Qs + r * D, Ks + key * (D + 1));
        const float p = rd[t] > 0.f ? expf(s - rm[t]) / rd[t] : 0.f;
        const float dp = dot<D>(dOs + r * D, Vs + key * (D + 1));
        DSs[r * KC + key] = p * (dp - dl[t]);
      }
      __syncthreads();
      for (int jj = 0; jj < KC; ++jj) {
        const float ds = DSs[orow * KC + jj];
        const float* krow = Ks + jj * (D + 1) + ocol;
#pragma unroll
        for (int i = 0; i < NO; ++i) acc[i] = fmaf(ds, krow[16 * i], acc[i]);
      }
    }
  }
  T* dQ = (T*)a.dQ + head + (size_t)(q0 + orow) * D + ocol;
#pragma unroll
  for (int i = 0; i < NO; ++i) dQ[16 * i] = from_f<T>(scale * acc[i]);
}

// ------------------------------------------------------------------ dK/dV --
// CTA = 16 key rows of block column n; warp w owns key rows 2w, 2w+1 and the
// lanes run over a chunk of QC queries of each block row that attends to n.
template <typename T, int D, int QC>
__global__ void __launch_bounds__(kThreads) dkdv_simt_kernel(BwdArgs a) {
  constexpr int KR = kRowsPerCta;
  constexpr int PER = 2 * QC / 32;
  constexpr int NO = D / 16;
  extern __shared__ float sm[];
  float* Kr = sm;                   // [KR][D]
  float* Vr = Kr + KR * D;          // [KR][D]
  float* Qs = Vr + KR * D;          // [QC][D+1]
  float* dOs = Qs + QC * (D + 1);   // [QC][D+1]
  float* Ps = dOs + QC * (D + 1);   // [KR][QC]
  float* DSs = Ps + KR * QC;        // [KR][QC]
  float* qm = DSs + KR * QC;        // [QC] row_max
  float* ql = qm + QC;              // [QC] row_denom
  float* qd = ql + QC;              // [QC] delta

  const int subs = kBlock / KR;
  const int n = blockIdx.x / subs;
  const int k0 = n * kBlock + (blockIdx.x % subs) * KR;
  const int bh = blockIdx.y;
  const size_t head = (size_t)bh * a.d.S * D;
  const T* Q = (const T*)a.Q + head;
  const T* dO = (const T*)a.dO + head;
  const float scale = a.d.scale;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int orow = threadIdx.x / 16, ocol = threadIdx.x % 16;

  load_rows<T, D>(Kr, D, (const T*)a.K + head + (size_t)k0 * D, KR);
  load_rows<T, D>(Vr, D, (const T*)a.V + head + (size_t)k0 * D, KR);

  float acc_k[NO], acc_v[NO];
#pragma unroll
  for (int i = 0; i < NO; ++i) { acc_k[i] = 0.f; acc_v[i] = 0.f; }

  const int t0 = a.col_ptr[n], t1 = a.col_ptr[n + 1];
  for (int t = t0; t < t1; ++t) {
    const int m = a.row_idx[t];
    if (bad_block(m, a.d.nb, a.status)) continue;
    for (int qc = 0; qc < kBlock; qc += QC) {
      const int i0 = m * kBlock + qc;
      __syncthreads();
      load_rows<T, D>(Qs, D + 1, Q + (size_t)i0 * D, QC);
      load_rows<T, D>(dOs, D + 1, dO + (size_t)i0 * D, QC);
      if (threadIdx.x < QC) {
        const size_t row = (size_t)bh * a.d.S + i0 + threadIdx.x;
        qm[threadIdx.x] = a.row_max[row];
        ql[threadIdx.x] = a.row_denom[row];
        qd[threadIdx.x] = a.delta[row];
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int e = lane + 32 * u;
        const int kr = 2 * warp + e / QC, qi = e % QC;
        const float s = scale * dot<D>(Kr + kr * D, Qs + qi * (D + 1));
        const float p = ql[qi] > 0.f ? expf(s - qm[qi]) / ql[qi] : 0.f;
        const float dp = dot<D>(Vr + kr * D, dOs + qi * (D + 1));
        Ps[kr * QC + qi] = p;
        DSs[kr * QC + qi] = p * (dp - qd[qi]);
      }
      __syncthreads();
      for (int ii = 0; ii < QC; ++ii) {
        const float p = Ps[orow * QC + ii];
        const float ds = DSs[orow * QC + ii];
        const float* gro = dOs + ii * (D + 1) + ocol;
        const float* qro = Qs + ii * (D + 1) + ocol;
#pragma unroll
        for (int i = 0; i < NO; ++i) {
          acc_v[i] = fmaf(p, gro[16 * i], acc_v[i]);
          acc_k[i] = fmaf(ds, qro[16 * i], acc_k[i]);
        }
      }
    }
  }
  T* dK = (T*)a.dK + head + (size_t)(k0 + orow) * D + ocol;
  T* dV = (T*)a.dV + head + (size_t)(k0 + orow) * D + ocol;
#pragma unroll
  for (int i = 0; i < NO; ++i) {
    dK[16 * i] = from_f<T>(scale * acc_k[i]);
    dV[16 * i] = from_f<T>(acc_v[i]);
  }
}

// ---------------------------------------------------------------- launch --
template <int D>
constexpr int chunk() { return D >= 512 ? 16 : 32; }

template <typename Kern>
bsr_status launch(Kern kern, dim3 grid, size_t smem, cudaStream_t s, const char* name, const void* args) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: cudaFuncSetAttribute: %s", name, cudaGetErrorString(e));
  }
  {
    LaunchTimer timer(name, s);
    void* argv[] = {const_cast<void*>(args)};
    cudaError_t e = cudaLaunchKernel((const void*)kern, grid, dim3(kThreads), argv, smem, s);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: launch: %s", name, cudaGetErrorString(e));
  }
  return BSR_OK;
}

template <typename T, int D>
bsr_status fwd_dispatch(const FwdArgs& a, cudaStream_t s) {
  constexpr int KC = chunk<D>();
  const size_t smem = sizeof(float) * (kRowsPerCta * D + KC * (D + 1) + KC * D + kRowsPerCta * KC + 3 * kRowsPerCta);
  dim3 grid(a.d.nb * (kBlock / kRowsPerCta), a.d.BH);
  return launch(fwd_simt_kernel<T, D, KC>, grid, smem, s, "fwd_simt", &a);
}

template <typename T, int D>
bsr_status dq_dispatch(const BwdArgs& a, cudaStream_t s) {
  constexpr int KC = chunk<D>();
  const size_t smem = sizeof(float) * (2 * kRowsPerCta * D + 2 * KC * (D + 1) + kRowsPerCta * KC);
  dim3 grid(a.d.nb * (kBlock / kRowsPerCta), a.d.BH);
  return launch(dq_simt_kernel<T, D, KC>, grid, smem, s, "dq_simt", &a);
}

template <typename T, int D>
bsr_status dkdv_dispatch(const BwdArgs& a, cudaStream_t s) {
  constexpr int QC = chunk<D>();
  const size_t smem = sizeof(float) * (2 * kRowsPerCta * D + 2 * QC * (D + 1) + 2 * kRowsPerCta * QC + 3 * QC);
  dim3 grid(a.d.nb * (kBlock / kRowsPerCta), a.d.BH);
  return launch(dkdv_simt_kernel<T, D, QC>, grid, smem, s, "dkdv_simt", &a);
}

template <typename T, int D>
bsr_status delta_dispatch(const BwdArgs& a, cudaStream_t s) {
  constexpr int G = D / 8 < 32 ? D / 8 : 32;
  const size_t rows = (size_t)a.d.BH * a.d.S;
  (void)G;
  const size_t groups = (rows + delta_rows_per_cta<T, D, kThreads>() - 1) / delta_rows_per_cta<T, D, kThreads>();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, delta_kernel<T, D>, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const size_t sms = (size_t)sm_count();
  const size_t resident = sms > 0 ? sms * per_sm : groups;
  dim3 grid((unsigned)(groups < resident ? groups : resident));
  return launch(delta_kernel<T, D>, grid, 0, s, "delta", &a);
}

#define BSR_DISPATCH_D(FN, T, ARGS, STREAM)                                      \
  do {                                                                          \
    switch ((ARGS).d.D) {                                                       \
      case 64: return FN<T, 64>(ARGS, STREAM);                                  \
      case 128: return FN<T, 128>(ARGS, STREAM);                                \
      case 256: return FN<T, 256>(ARGS, STREAM);                                \
      case 512: return FN<T, 512>(ARGS, STREAM);                                \
      default: return fail(BSR_ERR_UNSUPPORTED, "head_dim %d not supported", (ARGS).d.D); \
    }                                                                           \
  } while (0)

#define BSR_DISPATCH(FN, ARGS, STREAM)                                  \
  do {                                                                 \
    if ((ARGS).d.dtype == BSR_BF16) BSR_DISPATCH_D(FN, __nv_bfloat16, ARGS, STREAM); \
    if ((ARGS).d.dtype == BSR_F16) BSR_DISPATCH_D(FN, __half, ARGS, STREAM);         \
    BSR_DISPATCH_D(FN, float, ARGS, STREAM);                                         \
  } while (0)

}  // namespace

bsr_status launch_fwd_simt(const FwdArgs& a, cudaStream_t s) { BSR_DISPATCH(fwd_dispatch, a, s); }
bsr_status launch_delta(const BwdArgs& a, cudaStream_t s) { BSR_DISPATCH(delta_dispatch, a, s); }
bsr_status launch_dq_simt(const BwdArgs& a, cudaStream_t s) { BSR_DISPATCH(dq_dispatch, a, s); }
bsr_status launch_dkdv_simt(const BwdArgs& a, cudaStream_t s) { BSR_DISPATCH(dkdv_dispatch, a, s); }

}  // namespace bsr
