// Block-sparse times dense on the tensor cores (sm_103a): Y = A X for a
// static-structure BSR matrix A of 128 x 128 blocks (bf16 or fp16 values,
// fp32 accumulation) and a dense X ("trnsparse 0.7.0 -> 0.9.0" diff,
// CHANGELOG [0.8.0]: bsr_spmm_static walks exactly the stored blocks of
// each block row and addresses X by block column, with no padding to the
// longest row and no gather; CHANGELOG [0.9.0]: bf16 operands with fp32
// accumulation, one writer per output tile).
//
// One CTA per (block row m, column tile of NT columns of X / Y).  For each
// stored block j of row m, warp 0 loads the 128 x 128 block A_j (K-major,
// as stored) and the 128 x NT tile of X at block row col_idx[j] by TMA into
// a stage of a ring; lane 0 of warp 1 issues Y_m += A_j X_{col_idx[j]} as
// eight 128 x NT x 16 MMAs into TMEM; warps 2..5 (one output row per thread,
// its TMEM lane) round the accumulator to the operand type and store it.  A
// block row without stored blocks is written as zeros.  All waits are
// bounded (see sm100.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "sm100.cuh"
#include "tc_common.h"

namespace bsr {
namespace {

using namespace sm100;

constexpr int kSpmmThreads = 192;  // producer, MMA, 4 epilogue warps

template <int NT>
struct SpmmCfg {
  static constexpr int kATile = 128 * 128 * 2;  // one stored block
  static constexpr int kXTile = 128 * NT * 2;   // 128 rows of X, NT columns
  static constexpr int kStage = kATile + kXTile;
  static constexpr int kStages = NT == 64 ? 4 : 3;
  static constexpr int kBarOff = kStage * kStages;
  static constexpr int kSmem = kBarOff + 256;
};

struct SpmmBars {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t acc_full;  // every MMA of the tile is done
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(SpmmBars) <= 256, "barrier block overflows its shared-memory slot");

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

template <typename T, int NT>
__global__ void __launch_bounds__(kSpmmThreads, 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, SpmmArgs a) {
  using C = SpmmCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the 128-byte swizzle wants 1024-byte aligned tiles: refuse
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  SpmmBars* bars = (SpmmBars*)(smem_raw + C::kBarOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m = blockIdx.x;           // block row of A and Y
  const int n0 = blockIdx.y * NT;     // first column of the tile
  const int j0 = a.row_ptr[m], j1 = a.row_ptr[m + 1];
  const bool rows_ok = j0 >= 0 && j1 >= j0 && j1 <= a.nnzb;
  const int nblk = rows_ok ? j1 - j0 : 0;
  if (!rows_ok && threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->acc_full, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmX);
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int j = j0 + i;
        int k = a.col_idx[j];
        if (k < 0 || k >= a.n_bcols) {
          atomicExch(a.status, kStatusDeviceCheck);
          k = 0;
        }
        const int s = i % C::kStages;
        if (!mbar_wait(&bars->empty[s], ((i / C::kStages) & 1) ^ 1, ab, a.status)) break;
        uint8_t* st = smem_raw + s * C::kStage;
        mbar_arrive_expect_tx(&bars->full[s], C::kStage);
        for (int b = 0; b < 2; ++b) tma_load_2d(st + b * 16384, &tmA, b * 64, j * 128, &bars->full[s]);
        for (int b = 0; b < NT / 64; ++b)
          tma_load_2d(st + C::kATile + b * 16384, &tmX, n0 + b * 64, k * 128, &bars->full[s]);
        issued = i + 1;
      }
      // every copy issued has landed before the CTA exits
      for (int i = (issued > C::kStages ? issued - C::kStages : 0); i < issued; ++i)
        drain(&bars->full[i % C::kStages], (i / C::kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && nblk > 0) {
      // ----------------------------------------------------------- MMA --
      const uint32_t idesc = instr_desc(Half16<T>::kFmt, 0, 1, NT, 128);
      bool ok = true;
      for (int i = 0; i < nblk && ok; ++i) {
        const int s = i % C::kStages;
        if (!(ok = mbar_wait(&bars->full[s], (i / C::kStages) & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem_raw + s * C::kStage);
        const SDesc dA(base, 16, 1024), dX(base + C::kATile, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem, dA.at((kk >> 2) * 16384 + (kk & 3) * 32), dX.at(kk * 2048), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->empty[s]);
      }
      // also on a timeout, so the epilogue's wait ends and TMEM is idle
      mma_commit(&bars->acc_full);
      drain(&bars->acc_full, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue --
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    T* yrow = (T*)a.Y + ((size_t)m * 128 + r) * (size_t)a.n_cols + n0;
    if (nblk == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 0; c < NT / 8; ++c) ((uint4*)yrow)[c] = z;
    } else if (__all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, ab, a.status))) {
      tc_fence_after();
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
        st_rows64(w, yrow + c * 64, (size_t)a.n_cols);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, NT);
}

template <typename T, int NT>
bsr_status launch_spmm(const SpmmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmX, cudaStream_t s) {
  using C = SpmmCfg<NT>;
  auto kern = spmm_tc_kernel<T, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "spmm_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer("spmm_tc", s);
  kern<<<dim3(a.n_brows, a.n_cols / NT), kSpmmThreads, C::kSmem, s>>>(tmA, tmX, a);
  return check_launch("spmm_tc launch");
}

}  // namespace

bsr_status launch_spmm_tc(const SpmmArgs& a, cudaStream_t s) {
  // A: the stored blocks as nnzb * 128 rows of 128; X: n_bcols * 128 rows of n_cols
  Dims da{1, a.nnzb * 128, 128, 0, a.dtype, 1.f};
  Dims dx{1, a.n_bcols * 128, a.n_cols, 0, a.dtype, 1.f};
  CUtensorMap tmA, tmX;
  bsr_status st = make_tensor_map(da, a.A, &tmA, "A blocks");
  if (st == BSR_OK) st = make_tensor_map(dx, a.X, &tmX, "X");
  if (st != BSR_OK) return st;
  // 128-column tiles when they fill the SMs, else 64-column ones (twice the CTAs)
  const int sms = sm_count();
  const bool wide = a.n_cols % 128 == 0 && (long long)a.n_brows * (a.n_cols / 128) >= (sms > 0 ? sms : 1);
  if (a.dtype == BSR_F16)
    return wide ? launch_spmm<__half, 128>(a, tmA, tmX, s) : launch_spmm<__half, 64>(a, tmA, tmX, s);
  return wide ? launch_spmm<__nv_bfloat16, 128>(a, tmA, tmX, s) : launch_spmm<__nv_bfloat16, 64>(a, tmA, tmX, s);
}

}  // namespace bsr
