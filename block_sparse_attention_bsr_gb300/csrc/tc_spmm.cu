// Block-sparse times dense on the tensor cores (sm_103a), and the fused
// screened SpMM.
//
//  * bsr_spmm: Y = A X for a static-structure BSR matrix A of 128 x 128
//    blocks (bf16 or fp16 values, fp32 accumulation) and a dense X
//    ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0]: bsr_spmm_static
//    walks exactly the stored blocks of each block row and addresses X by
//    block column, with no padding to the longest row and no gather;
//    CHANGELOG [0.9.0]: bf16 operands with fp32 accumulation, one writer per
//    output tile).
//  * bsr_screened_spmm: C = (A o M) B for a dense square A and the pair-bound
//    mask M[i, j] = (q_i q_j > t), q = sqrt(|diag|), t = sqrt(threshold), all
//    in fp32 ("trnsparse 0.7.0 -> 0.9.0" diff, docs: screened_spmm fuses the
//    Schwarz bound, the threshold mask and the matmul into one dispatch).  The
//    planning launch first classifies every 128 x 128 tile of A by the least and
//    largest bound of its rows and columns (fp32 multiplication is monotone
//    for these non-negative bounds, so the block decisions agree with the
//    element ones): skipped (every pair fails), kept whole (every pair
//    passes) or masked element by element, and lists the kept tiles of each
//    block row in BSR form; the walk then multiplies exactly those tiles,
//    masking the partial ones in shared memory before their MMAs.
//
// bsr_spmm runs one CTA per (block row, column tile): warp 0 loads each
// stored block and the matching 128 x NT tile of X by TMA into a ring, lane 0
// of warp 1 issues the eight 128 x NT x 16 MMAs per block into TMEM, warps
// 2..5 store Y.  (The persistent walk below, tried for bsr_spmm as well, was
// slower on uniform random structures: its planning launch costs more than
// the balance it buys there.)
//
// The screened product's tiles gather in the first block rows (the bounds
// decay along the diagonal), so it runs as a persistent walk: the attention
// kernels' schedule (sched.cuh, plan.cu) with the column tiles of the output
// in the role of the heads: one
// CTA per SM takes (block row, column tile) items longest first from a
// global queue, block rows longer than the per-CTA share are cut into
// chunks whose fp32 partial products the last chunk to finish sums (in chunk
// order, so results are deterministic).  Warp 0 loads each tile of A and the
// matching 128 x NT tile of X by TMA into a ring; lane 0 of warp 1 issues
// Y += A_j X_k as eight 128 x NT x 16 MMAs into one of two TMEM
// accumulators (an item accumulates while the previous item's epilogue
// reads the other); warps 2..5 (one output row per thread, its TMEM lane)
// mask the screened tiles that need it and store the result.  All waits
// are bounded (see sm100.cuh).

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

constexpr int kWalkThreads = 192;  // producer, MMA, 4 masking / epilogue warps
constexpr int kSpmmThreads = 192;  // producer, MMA, 4 epilogue warps
constexpr int kMaxBlocks = kScreenMaxBlocks;  // screened: n <= 65536

template <int NT>
struct WalkCfg {
  static constexpr int kATile = 128 * 128 * 2;  // one tile of A
  static constexpr int kXTile = 128 * NT * 2;   // 128 rows of X, NT columns
  static constexpr int kStage = kATile + kXTile;
  static constexpr int kStages = NT == 64 ? 4 : (NT == 128 ? 3 : 2);
  static constexpr int kQOff = kStage * kStages;  // screened: float [128], bounds of a tile's columns
  static constexpr int kBarOff = kQOff + 128 * 4;
  static constexpr int kSmem = kBarOff + 512;
  static constexpr uint32_t kTmemCols = 2 * NT;  // two accumulators
  static_assert(kSmem <= 232448, "shared memory over the per-CTA limit");
  static_assert(kTmemCols <= 512, "TMEM columns over the allocation");
};

struct WalkBars {
  uint64_t full[4];       // A and X tiles landed
  uint64_t ready[4];      // screened: the A tile is masked (or needs no mask) and visible to the tensor core
  uint64_t empty[4];      // the tile's MMAs are done
  uint64_t acc_full[2];   // by accumulator: every MMA of the item is done
  uint64_t acc_empty[2];  // by accumulator: the epilogue has read it
  uint64_t sync128;       // bounded sync of the 128 masking threads
  uint64_t merge_sync;    // the epilogue warpgroup's sync around a split row's merge
  uint64_t final_mma;
  RingSmem ring;
  int merge_flag;
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(WalkBars) <= 512, "barrier block overflows its shared-memory slot");

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

// ------------------------------------------------ bsr_spmm: one CTA per tile --
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

template <typename T, int NT>
__global__ void __launch_bounds__(kSpmmThreads, 1)
    spmm_tile_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, SpmmArgs a) {
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
bsr_status launch_spmm_tile(const SpmmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmX, cudaStream_t s) {
  using C = SpmmCfg<NT>;
  auto kern = spmm_tile_kernel<T, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "spmm_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer("spmm_tc", s);
  kern<<<dim3(a.n_brows, a.n_cols / NT), kSpmmThreads, C::kSmem, s>>>(tmA, tmX, a);
  return check_launch("spmm_tc launch");
}

// ------------------------------------------- the persistent walk (screened) --
template <typename T, int NT, bool kScreen>
__global__ void __launch_bounds__(kWalkThreads, 1)
    spmm_walk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, SpmmArgs a) {
  // may run as a programmatic dependent of the planner: the prologue touches
  // only shared memory and TMEM
  griddep_launch_dependents();
  using C = WalkCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the 128-byte swizzle wants 1024-byte aligned tiles: refuse
    griddep_wait();
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  float* qcol = (float*)(smem_raw + C::kQOff);
  WalkBars* bars = (WalkBars*)(smem_raw + C::kBarOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = a.n_cols / NT;  // column tiles: the planner's "heads"
  const PlanLayout lay = plan_layout(a.plan, a.n_brows, (int)gridDim.x, BH, a.n_bcols);
  if (warp == 0) plan_prefetch_l2(a.plan, plan_words(a.n_brows, (int)gridDim.x, BH, a.n_bcols));

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->ready[i], 128);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 128);
    }
    mbar_init(&bars->sync128, 128);
    mbar_init(&bars->merge_sync, 128);
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 1 + 4);  // MMA thread, the 4 epilogue warps
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const Walk walk = make_walk(lay, BH);
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->ring;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmX);
      int gi = 0;  // tiles issued
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int w;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &w, ab, a.status)) || w < 0) break;
        Cursor cur;
        walk.decode(w, cur);
        const int n0 = cur.bh * NT;
        for (int i = 0; i < cur.n; ++i, ++gi) {
          const int j = cur.first + i;
          int k = a.col_idx[j];
          if (k < 0 || k >= a.n_bcols) {
            atomicExch(a.status, kStatusDeviceCheck);
            k = 0;
          }
          const int s = gi % C::kStages;
          if (!(ok = mbar_wait(&bars->empty[s], ((gi / C::kStages) & 1) ^ 1, ab, a.status))) break;
          uint8_t* st = smem_raw + s * C::kStage;
          mbar_arrive_expect_tx(&bars->full[s], C::kStage);
          for (int b = 0; b < 2; ++b) {
            if constexpr (kScreen)
              tma_load_2d(st + b * 16384, &tmA, k * 128 + b * 64, cur.line * 128, &bars->full[s]);
            else
              tma_load_2d(st + b * 16384, &tmA, b * 64, j * 128, &bars->full[s]);
          }
          for (int b = 0; b < NT / 64; ++b)
            tma_load_2d(st + C::kATile + b * 16384, &tmX, n0 + b * 64, k * 128, &bars->full[s]);
        }
      }
      // every copy issued has landed before the CTA exits
      for (int i = (gi > C::kStages ? gi - C::kStages : 0); i < gi; ++i)
        drain(&bars->full[i % C::kStages], (i / C::kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA --
      const uint32_t idesc = instr_desc(Half16<T>::kFmt, 0, 1, NT, 128);
      int gi = 0, q = 0;  // tiles consumed, non-empty items
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int w;
        if (!(ok = ring_get(ring, t, &w, ab, a.status)) || w < 0) break;
        Cursor cur;
        walk.decode(w, cur);
        if (cur.n > 0) {
          const int buf = q & 1;
          // the accumulator's previous item has been read by the epilogue
          if (q >= 2 && !(ok = mbar_wait(&bars->acc_empty[buf], ((q - 2) >> 1) & 1, ab, a.status))) break;
          tc_fence_after();
          for (int i = 0; i < cur.n && ok; ++i, ++gi) {
            const int s = gi % C::kStages;
            if (!(ok = mbar_wait(&bars->full[s], (gi / C::kStages) & 1, ab, a.status))) break;
            if (kScreen && !(ok = mbar_wait(&bars->ready[s], (gi / C::kStages) & 1, ab, a.status))) break;
            tc_fence_after();
            const uint32_t base = smem_u32(smem_raw + s * C::kStage);
            const SDesc dA(base, 16, 1024), dX(base + C::kATile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + buf * NT, dA.at((kk >> 2) * 16384 + (kk & 3) * 32), dX.at(kk * 2048), idesc,
                     (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars->empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->acc_full[buf]);
          ++q;
        }
        ring_release(ring, t);
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(&bars->final_mma);
      drain(&bars->final_mma, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------- masking, then the epilogue --
    const int wl = warp % 4;
    const int r = wl * 32 + lane;  // row of the A tile / of the output block row
    const int tid = threadIdx.x - 64;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const float t_bound = a.t;
    int gi = 0, q = 0, sync_phase = 0, merge_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int w = -1;
      if (lane == 0) ok = ring_get(ring, t, &w, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!ok || w < 0) break;
      Cursor cur;
      walk.decode(w, cur);
      const int m = cur.line, n0 = cur.bh * NT;
      T* yrow = (T*)a.Y + ((size_t)m * 128 + r) * (size_t)a.n_cols + n0;
      if (cur.n == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int c = 0; c < NT / 8; ++c) ((uint4*)yrow)[c] = z;
        __syncwarp();
        if (lane == 0) ring_release(ring, t);
        continue;
      }
      if constexpr (kScreen) {
        const float qr = sqrtf(fabsf(a.diag[(size_t)m * 128 + r]));
        for (int i = 0; i < cur.n && ok; ++i, ++gi) {
          const int s = gi % C::kStages;
          const int j = cur.first + i;
          // every tile waits for its copy, so the ready arrivals of this
          // warpgroup never run a whole ring ahead of the MMA thread
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (gi / C::kStages) & 1, ab, a.status))))
            break;
          if (a.cls[j] == kTilePartial) {
            int k = a.col_idx[j];
            k = (k < 0 || k >= a.n_bcols) ? 0 : k;
            qcol[tid] = sqrtf(fabsf(a.diag[(size_t)k * 128 + tid]));
            if (!(ok = group_sync(&bars->sync128, sync_phase, ab, a.status))) break;
            // row r of the tile: 16-byte chunk c of box b (columns 64 b + 8 c ..)
            // sits at chunk position c ^ (r % 8) of the row (128-byte swizzle)
            const uint32_t row = smem_u32(smem_raw + s * C::kStage) + r * 128;
#pragma unroll 1
            for (int b = 0; b < 2; ++b) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint32_t addr = row + b * 16384 + ((c ^ (r & 7)) << 4);
                uint32_t v[4];
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                             : "r"(addr));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int col = b * 64 + c * 8 + 2 * e;
                  const uint32_t keep_lo = qr * qcol[col] > t_bound ? 0x0000ffffu : 0u;
                  const uint32_t keep_hi = qr * qcol[col + 1] > t_bound ? 0xffff0000u : 0u;
                  v[e] &= keep_lo | keep_hi;
                }
                st_shared_v4(addr, v[0], v[1], v[2], v[3]);
              }
            }
            fence_proxy_async_smem();
            // qcol is rewritten for the next partial tile
            if (!(ok = group_sync(&bars->sync128, sync_phase, ab, a.status))) break;
          }
          mbar_arrive(&bars->ready[s]);
        }
        if (!ok) break;
      }
      const int buf = q & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full[buf], (q >> 1) & 1, ab, a.status)))) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + buf * NT;
      if (cur.slot < 0) {
#pragma unroll 1
        for (int c = 0; c < NT / 64; ++c) {
          uint32_t v[32], u[32];
          tmem_ld32(tacc + c * 64, v);
          tmem_ld32(tacc + c * 64 + 32, u);
          tmem_wait_ld();
          uint32_t o[32];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            o[x] = Half16<T>::pack(__uint_as_float(v[2 * x]), __uint_as_float(v[2 * x + 1]));
            o[16 + x] = Half16<T>::pack(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1]));
          }
          st_rows64(o, yrow + c * 64, (size_t)a.n_cols);
        }
      } else {
        // chunk of a split row: publish the fp32 partial product, the last
        // chunk of the row (for this column tile) sums them all in order
        const size_t kTileF = (size_t)128 * NT;
        store_acc_part<NT>(tacc, a.part + ((size_t)cur.slot * BH + cur.bh) * kTileF, 0, r);
        bool last = false;
        if (!(ok = merge_arrive(lay, cur.slot, cur.bh, BH, 0, r, &bars->merge_flag, &bars->merge_sync, merge_phase,
                                ab, a.status, &last)))
          break;
        if (last) {
          const int sl = lay.slot_line[cur.slot];
          const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
          merge_tiles<NT>(a.part + ((size_t)base * BH + cur.bh) * kTileF, (size_t)BH * kTileF, nc, 0, r, yrow, 1.f);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[buf]);
      ++q;
      __syncwarp();
      if (lane == 0) ring_release(ring, t);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0) plan_exit(lay);
}

// Column tile width: the widest of 256 / 128 / 64 that divides n_cols and
// still gives every SM an item (wider tiles run wider MMAs), else 64.
int walk_nt(int n_brows, int n_cols) {
  const long long sms = sm_count() > 0 ? sm_count() : 1;
  for (int nt = 256; nt >= 128; nt /= 2)
    if (n_cols % nt == 0 && (long long)n_brows * (n_cols / nt) >= sms) return nt;
  return 64;
}

// The persistent grid: one CTA per SM (split rows make more items than
// rows), at most one per (block row, column tile) times the split factor
// the planner allows.
int walk_grid(int n_brows, int n_cols) {
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const long long work = (long long)n_brows * (n_cols / walk_nt(n_brows, n_cols)) * 8;
  return (int)(work < sms ? work : sms);
}

size_t walk_scratch_bytes(int n_brows, int n_bcols, int n_cols, int G) {
  const int NT = walk_nt(n_brows, n_cols), BH = n_cols / NT;
  return sizeof(int32_t) * plan_words(n_brows, G, BH, n_bcols) +
         sizeof(float) * (size_t)128 * NT * plan_tiles(n_brows, G, BH, n_bcols);
}

template <typename T, int NT, bool kScreen>
bsr_status launch_walk_nt(const SpmmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmX, int G,
                          cudaStream_t s) {
  using C = WalkCfg<NT>;
  auto kern = spmm_walk_kernel<T, NT, kScreen>;
  const char* name = kScreen ? "screened_tc" : "spmm_tc";
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: cudaFuncSetAttribute(%d): %s", name, C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer(name, s);
  e = launch_dependent(kern, dim3(G), dim3(kWalkThreads), C::kSmem, s, tmA, tmX, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

// Plans the rows of a (split into chunks, column tiles as heads) in
// `scratch` and launches the walk.
template <bool kScreen>
bsr_status run_walk(SpmmArgs a, const CUtensorMap& tmA, const CUtensorMap& tmX, void* scratch, cudaStream_t s,
                    const ScreenListArgs* list = nullptr) {
  const int NT = walk_nt(a.n_brows, a.n_cols), BH = a.n_cols / NT;
  const int G = walk_grid(a.n_brows, a.n_cols);
  if (G <= 0) return fail(BSR_ERR_CUDA, "spmm: cannot query the SM count");
  a.plan = (int32_t*)scratch;
  a.part = (float*)((char*)scratch + sizeof(int32_t) * plan_words(a.n_brows, G, BH, a.n_bcols));
  PlanArgs p{};
  p.list[0] = PlanList{a.row_ptr, a.plan};
  p.n = a.n_brows;
  p.max_len = a.n_bcols;  // a block row may store up to n_bcols blocks
  p.G = G;
  p.BH = BH;
  p.allow_split = 1;
  p.status = a.status;
  // the screened product builds its tile list in the planner's launch
  bsr_status st = list ? launch_screen_plan(*list, p, s) : launch_plan(p, 1, s);
  if (st != BSR_OK) return st;
  const bool f16 = a.dtype == BSR_F16;
  switch (NT) {
    case 256:
      return f16 ? launch_walk_nt<__half, 256, kScreen>(a, tmA, tmX, G, s)
                 : launch_walk_nt<__nv_bfloat16, 256, kScreen>(a, tmA, tmX, G, s);
    case 128:
      return f16 ? launch_walk_nt<__half, 128, kScreen>(a, tmA, tmX, G, s)
                 : launch_walk_nt<__nv_bfloat16, 128, kScreen>(a, tmA, tmX, G, s);
    default:
      return f16 ? launch_walk_nt<__half, 64, kScreen>(a, tmA, tmX, G, s)
                 : launch_walk_nt<__nv_bfloat16, 64, kScreen>(a, tmA, tmX, G, s);
  }
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
    return wide ? launch_spmm_tile<__half, 128>(a, tmA, tmX, s) : launch_spmm_tile<__half, 64>(a, tmA, tmX, s);
  return wide ? launch_spmm_tile<__nv_bfloat16, 128>(a, tmA, tmX, s) : launch_spmm_tile<__nv_bfloat16, 64>(a, tmA, tmX, s);
}


bsr_status launch_screened_tc(const ScreenedArgs& sa, cudaStream_t s) {
  const int nb = sa.n / 128;
  if (nb > kMaxBlocks) return fail(BSR_ERR_UNSUPPORTED, "screened_spmm: n %d above %d", sa.n, kMaxBlocks * 128);
  Dims da{1, sa.n, sa.n, 0, sa.dtype, 1.f};
  Dims db{1, sa.n, sa.n_cols, 0, sa.dtype, 1.f};
  CUtensorMap tmA, tmB;
  bsr_status st = make_tensor_map(da, sa.A, &tmA, "A");
  if (st == BSR_OK) st = make_tensor_map(db, sa.B, &tmB, "B");
  if (st != BSR_OK) return st;
  const int G = walk_grid(nb, sa.n_cols);
  if (G <= 0) return fail(BSR_ERR_CUDA, "screened_spmm: cannot query the SM count");
  // scratch: the tile list (row_ptr, col_idx, class), then the plan and partial tiles
  const size_t list_ints = (size_t)(nb + 1 + 3) / 4 * 4 + 2 * (size_t)nb * nb;
  const size_t list_bytes = sizeof(int32_t) * ((list_ints + 3) / 4 * 4);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, list_bytes + walk_scratch_bytes(nb, nb, sa.n_cols, G), s);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "screened_spmm: cudaMallocAsync: %s", cudaGetErrorString(e));
  ScreenListArgs la{};
  la.diag = sa.diag;
  la.nb = nb;
  la.t = sqrtf(sa.threshold);
  la.row_ptr = (int32_t*)scratch;
  la.col_idx = la.row_ptr + (size_t)(nb + 1 + 3) / 4 * 4;
  la.cls = la.col_idx + (size_t)nb * nb;
  SpmmArgs a{};
  a.A = sa.A;
  a.X = sa.B;
  a.Y = sa.C;
  a.row_ptr = la.row_ptr;
  a.col_idx = la.col_idx;
  a.n_brows = nb;
  a.n_bcols = nb;
  a.nnzb = nb * nb;
  a.n_cols = sa.n_cols;
  a.dtype = sa.dtype;
  a.status = sa.status;
  a.cls = la.cls;
  a.diag = sa.diag;
  a.t = la.t;
  st = run_walk<true>(a, tmA, tmB, (char*)scratch + list_bytes, s, &la);
  e = cudaFreeAsync(scratch, s);
  if (st == BSR_OK && e != cudaSuccess) st = fail(BSR_ERR_CUDA, "screened_spmm: cudaFreeAsync: %s", cudaGetErrorString(e));
  return st;
}

}  // namespace bsr
