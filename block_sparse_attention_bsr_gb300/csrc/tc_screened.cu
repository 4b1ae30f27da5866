// Fused screened SpMM on the tensor cores (sm_103a): C = (A o M) B for a
// dense square A (n x n) and dense B (n x n_cols), with the pair-bound mask
// M[i, j] = (q_i q_j > t), q = sqrt(|diag|), t = sqrt(threshold), all in
// fp32 ("trnsparse 0.7.0 -> 0.9.0" diff, docs: screened_spmm(A, diag, B,
// threshold) fuses the Schwarz bound, the threshold mask and the matmul
// into one dispatch; the mask semantics are stated there).
//
// One CTA per (128-row block m, column tile of NT columns).  Every thread
// first computes, for each 128-column block k of A, the least and largest
// bound q over its columns (block m's row bounds are the same numbers, A
// being square).  A tile (m, k) is then
//   * skipped when max_m * max_k <= t (every pair fails),
//   * multiplied as loaded when min_m * min_k > t (every pair passes),
//   * otherwise masked element by element in shared memory first.
// fp32 multiplication is monotone for these non-negative bounds, so the
// block decisions agree with the element ones.  Warp 0 loads the kept
// tiles of A and the matching 128-row tiles of B by TMA into a ring;
// warps 2..5 (one A row per thread) mask the tiles that need it, make the
// writes visible to the tensor core and hand every kept tile on; lane 0 of
// warp 1 issues the 128 x NT x 16 MMAs into TMEM; warps 2..5 store C.
// All waits are bounded (see sm100.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.h"
#include "sched.cuh"
#include "sm100.cuh"
#include "tc_common.h"

namespace bsr {
namespace {

using namespace sm100;

constexpr int kScrThreads = 192;  // producer, MMA, 4 warps for bounds / masking / epilogue
constexpr int kMaxBlocks = 512;   // n <= 65536

template <int NT>
struct ScrCfg {
  static constexpr int kATile = 128 * 128 * 2;
  static constexpr int kBTile = 128 * NT * 2;
  static constexpr int kStage = kATile + kBTile;
  static constexpr int kStages = NT == 64 ? 4 : 3;
  static constexpr int kBoundOff = kStage * kStages;              // float2 [n / 128]: (min q, max q)
  static constexpr int kQColOff = kBoundOff + kMaxBlocks * 8;     // float [128]: q of the tile's columns
  static constexpr int kBarOff = kQColOff + 128 * 4;
  static constexpr int kSmem = kBarOff + 256;
};

struct ScrBars {
  uint64_t full[4];    // A and B tiles landed
  uint64_t ready[4];   // the A tile is masked (or needs no mask) and visible to the tensor core
  uint64_t empty[4];   // the tile's MMAs are done
  uint64_t acc_full;
  uint64_t sync128;    // bounded sync of the 128 masking threads (group_sync)
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(ScrBars) <= 256, "barrier block overflows its shared-memory slot");

enum : int { kSkip = 0, kFull = 1, kPartial = 2 };

__device__ __forceinline__ float bound_of(const float* diag, int i) { return sqrtf(fabsf(diag[i])); }

__device__ __forceinline__ int tile_class(float2 row, float2 col, float t) {
  if (!(row.y * col.y > t)) return kSkip;
  return row.x * col.x > t ? kFull : kPartial;
}

__device__ __forceinline__ void drain_scr(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

template <typename T, int NT>
__global__ void __launch_bounds__(kScrThreads, 1)
    screened_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       ScreenedArgs a) {
  using C = ScrCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the 128-byte swizzle wants 1024-byte aligned tiles: refuse
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  float2* bnd = (float2*)(smem_raw + C::kBoundOff);
  float* qcol = (float*)(smem_raw + C::kQColOff);
  ScrBars* bars = (ScrBars*)(smem_raw + C::kBarOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nb = a.n / 128;
  const int m = blockIdx.x;
  const int n0 = blockIdx.y * NT;
  const float t = sqrtf(a.threshold);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->ready[i], 128);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->sync128, 128);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, NT);
    tmem_relinquish();
  }
  // bounds of every 128-column block: thread x takes blocks x, x + 192, ...
  // (32 independent 16-byte loads of the block's 128 values in flight)
  for (int k = threadIdx.x; k < nb; k += kScrThreads) {
    const float4* d = (const float4*)(a.diag + (size_t)k * 128);
    float lo = INFINITY, hi = 0.f;
#pragma unroll 8
    for (int v = 0; v < 32; ++v) {
      const float4 x = d[v];
      const float q0 = sqrtf(fabsf(x.x)), q1 = sqrtf(fabsf(x.y)), q2 = sqrtf(fabsf(x.z)), q3 = sqrtf(fabsf(x.w));
      lo = fminf(lo, fminf(fminf(q0, q1), fminf(q2, q3)));
      hi = fmaxf(hi, fmaxf(fmaxf(q0, q1), fmaxf(q2, q3)));
    }
    bnd[k] = make_float2(lo, hi);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  const float2 rowb = bnd[m];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int i = 0;
      for (int k = 0; k < nb; ++k) {
        if (tile_class(rowb, bnd[k], t) == kSkip) continue;
        const int s = i % C::kStages;
        if (!mbar_wait(&bars->empty[s], ((i / C::kStages) & 1) ^ 1, ab, a.status)) break;
        uint8_t* st = smem_raw + s * C::kStage;
        mbar_arrive_expect_tx(&bars->full[s], C::kStage);
        for (int b = 0; b < 2; ++b) tma_load_2d(st + b * 16384, &tmA, k * 128 + b * 64, m * 128, &bars->full[s]);
        for (int b = 0; b < NT / 64; ++b)
          tma_load_2d(st + C::kATile + b * 16384, &tmB, n0 + b * 64, k * 128, &bars->full[s]);
        ++i;
      }
      for (int x = (i > C::kStages ? i - C::kStages : 0); x < i; ++x)
        drain_scr(&bars->full[x % C::kStages], (x / C::kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA --
      const uint32_t idesc = instr_desc(Half16<T>::kFmt, 0, 1, NT, 128);
      int i = 0;
      bool ok = true;
      for (int k = 0; k < nb && ok; ++k) {
        if (tile_class(rowb, bnd[k], t) == kSkip) continue;
        const int s = i % C::kStages;
        // the tiles landed (this thread's own view of the copies) and the A
        // tile is masked; the stage is refilled only after this thread's
        // commit, so neither phase can run ahead
        if (!(ok = mbar_wait(&bars->full[s], (i / C::kStages) & 1, ab, a.status))) break;
        if (!(ok = mbar_wait(&bars->ready[s], (i / C::kStages) & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem_raw + s * C::kStage);
        const SDesc dA(base, 16, 1024), dB(base + C::kATile, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem, dA.at((kk >> 2) * 16384 + (kk & 3) * 32), dB.at(kk * 2048), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->empty[s]);
        ++i;
      }
      // also after a timeout, so the epilogue's wait ends and TMEM is idle
      mma_commit(&bars->acc_full);
      drain_scr(&bars->acc_full, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------- masking, then the epilogue --
    const int wl = warp % 4;
    const int r = wl * 32 + lane;  // row of the A tile / of C in this block
    const int tid = threadIdx.x - 64;
    const float qr = bound_of(a.diag, m * 128 + r);
    int i = 0, phase = 0;
    bool ok = true;
    for (int k = 0; k < nb && ok; ++k) {
      const int cls = tile_class(rowb, bnd[k], t);
      if (cls == kSkip) continue;
      const int s = i % C::kStages;
      if (cls == kPartial) {
        qcol[tid] = bound_of(a.diag, k * 128 + tid);
        if (!(ok = group_sync(&bars->sync128, phase, ab, a.status))) break;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (i / C::kStages) & 1, ab, a.status)))) break;
        // row r of the tile: 16-byte chunk c of box b (columns 64 b + 8 c ..)
        // sits at chunk position c ^ (r % 8) of the row (128-byte swizzle)
        const uint32_t row = smem_u32(smem_raw + s * C::kStage) + r * 128;
#pragma unroll 1
        for (int b = 0; b < 2; ++b) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t addr = row + b * 16384 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(addr));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = b * 64 + c * 8 + 2 * e;
              const uint32_t keep_lo = qr * qcol[j] > t ? 0x0000ffffu : 0u;
              const uint32_t keep_hi = qr * qcol[j + 1] > t ? 0xffff0000u : 0u;
              w[e] &= keep_lo | keep_hi;
            }
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        // qcol is rewritten for the next partial tile
        if (!(ok = group_sync(&bars->sync128, phase, ab, a.status))) break;
      } else {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (i / C::kStages) & 1, ab, a.status)))) break;
      }
      mbar_arrive(&bars->ready[s]);
      ++i;
    }
    T* crow = (T*)a.C + ((size_t)m * 128 + r) * (size_t)a.n_cols + n0;
    if (i == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 0; c < NT / 8; ++c) ((uint4*)crow)[c] = z;
    } else if (__all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, ab, a.status))) {
      tc_fence_after();
      const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
#pragma unroll 1
      for (int c = 0; c < NT / 64; ++c) {
        uint32_t v[32], u[32];
        tmem_ld32(tmem + lane_base + c * 64, v);
        tmem_ld32(tmem + lane_base + c * 64 + 32, u);
        tmem_wait_ld();
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          w[q] = Half16<T>::pack(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
          w[16 + q] = Half16<T>::pack(__uint_as_float(u[2 * q]), __uint_as_float(u[2 * q + 1]));
        }
        st_rows64(w, crow + c * 64, (size_t)a.n_cols);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, NT);
}

template <typename T, int NT>
bsr_status launch_screened(const ScreenedArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t s) {
  using C = ScrCfg<NT>;
  auto kern = screened_tc_kernel<T, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "screened_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer("screened_tc", s);
  kern<<<dim3(a.n / 128, a.n_cols / NT), kScrThreads, C::kSmem, s>>>(tmA, tmB, a);
  return check_launch("screened_tc launch");
}

}  // namespace

bsr_status launch_screened_tc(const ScreenedArgs& a, cudaStream_t s) {
  if (a.n / 128 > kMaxBlocks) return fail(BSR_ERR_UNSUPPORTED, "screened_spmm: n %d above %d", a.n, kMaxBlocks * 128);
  Dims da{1, a.n, a.n, 0, a.dtype, 1.f};
  Dims db{1, a.n, a.n_cols, 0, a.dtype, 1.f};
  CUtensorMap tmA, tmB;
  bsr_status st = make_tensor_map(da, a.A, &tmA, "A");
  if (st == BSR_OK) st = make_tensor_map(db, a.B, &tmB, "B");
  if (st != BSR_OK) return st;
  const int sms = sm_count();
  const bool wide = a.n_cols % 128 == 0 && (long long)(a.n / 128) * (a.n_cols / 128) >= (sms > 0 ? sms : 1);
  if (a.dtype == BSR_F16)
    return wide ? launch_screened<__half, 128>(a, tmA, tmB, s) : launch_screened<__half, 64>(a, tmA, tmB, s);
  return wide ? launch_screened<__nv_bfloat16, 128>(a, tmA, tmB, s)
              : launch_screened<__nv_bfloat16, 64>(a, tmA, tmB, s);
}

}  // namespace bsr
