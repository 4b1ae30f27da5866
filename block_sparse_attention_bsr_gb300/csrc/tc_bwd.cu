// Tensor-core backward pass for 16-bit operands (bf16 or fp16, fp32
// accumulation; head_dim 64 / 128, and the dQ walk over stored dS tiles at
// every head_dim) on sm_103a.
//
// Persistent kernels, each output tile with exactly one writer and no
// atomics ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.5.1]):
//
//  * dK/dV (column-first over the BSC lists, _attn_bwd_dkdv_kernel): work
//    items are block columns n of one (batch, head).  For every block row m
//    that stores (m, n):
//        S^T = K_n Q_m^T,  dP^T = V_n dO_m^T                 (tcgen05, TMEM)
//        P^T = exp(scale S^T - row_max) / row_denom,  dS^T = P^T * (dP^T - D_m)
//        dV_n += P^T dO_m,   dK_n += dS^T Q_m                  (tcgen05, TMEM)
//    and dK_n * scale, dV_n are stored at the end.  On a plan it also stores
//    each dS tile (bf16 / fp16) for the dQ walk below.
//  * dQ over stored dS (row-first, on a plan): items are block rows m; for
//    every stored block (m, n), dQ_m += dS_mn K_n, and dQ_m * scale is
//    stored at the end (dq_ds_kernel).
//  * dQ recomputing (row-first, mirrors the forward, _attn_bwd_dq_kernel; the
//    per-call entry points): for every stored block (m, n)
//        S  = Q_m K_n^T,  dP = dO_m V_n^T,  P and dS as above,  dQ_m += dS K_n.
//
// The statistics enter as one base-2 log-sum-exp per query,
// lse2 = row_max log2(e) + log2(row_denom), so P = 2^(scale log2(e) S - lse2);
// lse2 and the delta D_i = dO_i . O_i ("trnsparse 0.4.1 -> 0.6.0" diff,
// CHANGELOG [0.5.0]) come from the delta kernel that runs first.
//
// Warp roles of the dK/dV and recomputing dQ kernels (320 threads): warp 0
// TMA producer, warp 1 TMEM owner and MMA issuer, warps 2..9 two elementwise
// warpgroups.  Thread (warp w, lane l) owns TMEM lane 32 (w % 4) + l (a query
// row in dQ, a key row in dK/dV); warpgroup g = (w - 2) / 4 handles columns
// [64 g, 64 g + 64) of the 128 x 128 score tiles and half of the output
// columns in the epilogue.  A warpgroup copies its S / dP columns into
// registers at once and releases them, so the MMA of the next block overlaps
// the elementwise work of this one.  dS (dQ kernel), P^T and dS^T (dK/dV
// kernel) go back to TMEM as 16-bit values and feed the next MMA as its A
// operand from TMEM.  All waits are bounded (see sm100.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"
#include "sched.cuh"
#include "sm100.cuh"
#include "tc_common.h"

namespace bsr {
namespace {

using namespace sm100;

constexpr int kThreads = 320;
constexpr int kEw = 256;  // elementwise threads
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Drains: polls `bar` for the phase of parity `parity` for at most 0.2 s.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

// Stores NC fp32 TMEM columns of this thread's lane (from taddr) as T
// times `mul` to global memory at grow (the warp's 32 lanes hold 32
// consecutive rows, ld elements apart): 64 columns per round, both 32-column
// loads in flight before the one wait, rows exchanged in groups of four so
// the stores cover whole 128-byte lines (st_rows64).
template <int NC, typename T>
__device__ __forceinline__ void store_acc_cols(uint32_t taddr, T* grow, float mul, size_t ld) {
  static_assert(NC % 32 == 0, "whole 32-column loads");
#pragma unroll 1
  for (int c = 0; c < NC / 64; ++c) {
    uint32_t v[32], u[32];
    tmem_ld32(taddr + c * 64, v);
    tmem_ld32(taddr + c * 64 + 32, u);
    tmem_wait_ld();
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      w[j] = Half16<T>::pack(__uint_as_float(v[2 * j]) * mul, __uint_as_float(v[2 * j + 1]) * mul);
      w[16 + j] = Half16<T>::pack(__uint_as_float(u[2 * j]) * mul, __uint_as_float(u[2 * j + 1]) * mul);
    }
    st_rows64(w, grow + c * 64, ld);
  }
  if constexpr (NC % 64 != 0) {
    uint32_t v[32];
    tmem_ld32(taddr + NC - 32, v);
    tmem_wait_ld();
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = Half16<T>::pack(__uint_as_float(v[2 * j]) * mul, __uint_as_float(v[2 * j + 1]) * mul);
    st_global_64B(grow + NC - 32, w);
  }
}

template <int NC, typename T>
__device__ __forceinline__ void zero_cols(T* grow) {
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int c = 0; c < NC / 8; ++c) ((uint4*)grow)[c] = z;
}

// Packs 64 fp32 values to pairs of T and stores them in 32 TMEM columns.
template <typename T>
__device__ __forceinline__ void tmem_st_pairs64(uint32_t taddr, const float (&x)[64]) {
  uint32_t v[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = Half16<T>::pack(x[2 * k], x[2 * k + 1]);
  tmem_st32(taddr, v);
}

// =================================================================== dQ ====
template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  // K_g is held until dQ_g (the last MMA of block g) and is needed again
  // right after it, so it gets one stage more than V.
  static constexpr int kKStages = D == 64 ? 4 : 3;
  static constexpr int kVStages = D == 64 ? 4 : 2;
  static constexpr int kBarOff = kTile * (2 + kKStages + kVStages);
  static constexpr int kSmem = kBarOff + 512 + 1024;
};

struct DqBars {
  uint64_t qd_full;
  uint64_t qd_empty;
  uint64_t sdp_full;
  uint64_t sdp_free;
  // by dS buffer, like dq_done: with two buffers the elementwise pass may run
  // two blocks ahead of the MMA thread, so one barrier could alias phases
  uint64_t ds_full[2];
  uint64_t dq_done[2];  // by dS buffer: dQ of a block that read it is done
  uint64_t final_mma;
  uint64_t wg_sync[2];
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  RingSmem ring;
  int merge_flag[2];
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 512, "barrier block overflows its shared-memory slot");

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, BwdArgs a) {
  // may run as a programmatic dependent: the prologue below touches only
  // shared memory and TMEM; global memory waits for the previous grid
  griddep_launch_dependents();
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sdO = sQ + C::kTile;
  uint8_t* sK = sdO + C::kTile;
  uint8_t* sV = sK + C::kKStages * C::kTile;
  DqBars* bars = (DqBars*)(sm + C::kBarOff);
  // dS (bf16) of block g at column 384 + 64 (g % 2): two buffers, so the
  // elementwise pass of block g waits only for dQ of block g - 2
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
  static_assert(kColDQ + D <= kColDS && kColDS + 2 * 64 <= kTmemCols, "TMEM columns over the allocation");
  static_assert(C::kSmem <= 232448, "shared memory over the per-CTA limit");

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const PlanLayout lay = plan_layout(a.row_plan, a.d.nb, (int)gridDim.x, a.d.BH);
  if (warp == 0) plan_prefetch_l2(a.row_plan, plan_words(a.d.nb, (int)gridDim.x, a.d.BH));

  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 1);
    mbar_init(&bars->qd_empty, 1);
    mbar_init(&bars->sdp_full, 1);
    mbar_init(&bars->sdp_free, kEw);
    mbar_init(&bars->ds_full[0], kEw);
    mbar_init(&bars->ds_full[1], kEw);
    mbar_init(&bars->dq_done[0], 1);
    mbar_init(&bars->dq_done[1], 1);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->wg_sync[0], 128);
    mbar_init(&bars->wg_sync[1], 128);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 1 + kEw / 32);  // MMA thread + elementwise warps
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const Walk walk = make_walk(lay, a.d.BH);
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->ring;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      int g = 0, q = 0, kg = 0, vg = 0;
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        if (cur.n == 0) continue;
        // Q, dO of a new item: the previous item's S / dP MMAs must be done
        if (!(ok = mbar_wait(&bars->qd_empty, (q & 1) ^ 1, ab, a.status))) break;
        const int qrow = cur.bh * S + cur.line * 128;
        mbar_arrive_expect_tx(&bars->qd_full, 2 * C::kTile);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_2d(sQ + b * 16384, &tmQ, b * 64, qrow, &bars->qd_full);
          tma_load_2d(sdO + b * 16384, &tmdO, b * 64, qrow, &bars->qd_full);
        }
        ++q;
        for (int i = 0; i < cur.n; ++i, ++g) {
          int n = a.col_idx[cur.first + i];
          if (n < 0 || n >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            n = 0;
          }
          const int krow = cur.bh * S + n * 128;
          const int ks = g % C::kKStages, vs = g % C::kVStages;
          if (!(ok = mbar_wait(&bars->k_empty[ks], ((g / C::kKStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->k_full[ks], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sK + ks * C::kTile + b * 16384, &tmK, b * 64, krow, &bars->k_full[ks]);
          kg = g + 1;
          if (!(ok = mbar_wait(&bars->v_empty[vs], ((g / C::kVStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->v_full[vs], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sV + vs * C::kTile + b * 16384, &tmV, b * 64, krow, &bars->v_full[vs]);
          vg = g + 1;
        }
      }
      // drain: every copy issued must land before the CTA exits
      if (q > 0) drain_wait(&bars->qd_full, (q - 1) & 1);
      for (int i = (kg > C::kKStages ? kg - C::kKStages : 0); i < kg; ++i)
        drain_wait(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1);
      for (int i = (vg > C::kVStages ? vg - C::kVStages : 0); i < vg; ++i)
        drain_wait(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1);
    }
  } else if (warp == 1) {
    {
      // ----------------------------------------------------------- MMA --
      // The whole warp walks the schedule (descriptor arithmetic stays
      // warp-uniform); one elected lane issues the MMAs and commits.
      const uint32_t leader = elect_one();
      // S / dP of block g+1 (cursor A) are issued before dQ of block g
      // (cursor B), so they run while the elementwise pass of block g
      // computes dS.  A draws items from the ring; B follows and releases
      // each item once it is past it.
      const uint32_t idS = instr_desc(Half16<T>::kFmt, 0, 0, 128, 128);
      const uint32_t idDQ = instr_desc(Half16<T>::kFmt, 0, 1, D, 128);
      const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = true;
      auto seek_a = [&](Cursor& c) {
        while (true) {
          int k;
          int kk0 = -1;
          bool good = true;
          if (lane == 0) good = ring_get(ring, c.t, &kk0, ab, a.status);
          ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
          k = __shfl_sync(0xffffffffu, kk0, 0);
          if (!ok || k < 0) {
            c.done = true;
            return;
          }
          walk.decode(k, c);
          if (c.n > 0) {
            c.i = 0;
            return;
          }
          ++c.t;
        }
      };
      auto seek_b = [&](Cursor& c) {
        while (true) {
          const int k = *(volatile int32_t*)&ring->k[c.t % kRing];
          if (k < 0) {
            c.done = true;
            return;
          }
          walk.decode(k, c);
          if (c.n > 0) {
            c.i = 0;
            return;
          }
          __syncwarp();
          if (lane == 0) ring_release(ring, c.t);
          ++c.t;
        }
      };
      auto issue_sdp = [&](const Cursor& c) -> bool {
        const int ks = c.g % C::kKStages, vs = c.g % C::kVStages;
        if (c.i == 0 && !warp_wait(&bars->qd_full, c.q & 1, ab, a.status)) return false;
        if (!warp_wait(&bars->k_full[ks], (c.g / C::kKStages) & 1, ab, a.status)) return false;
        if (!warp_wait(&bars->v_full[vs], (c.g / C::kVStages) & 1, ab, a.status)) return false;
        if (!warp_wait(&bars->sdp_free, (c.g & 1) ^ 1, ab, a.status)) return false;
        tc_fence_after();
        const SDesc dQ(aQ, 16, 1024), dO(adO, 16, 1024), dK(aK + ks * C::kTile, 16, 1024),
            dV(aV + vs * C::kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_by(leader, tmem + kColS, dQ.at(off), dK.at(off), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_by(leader, tmem + kColDP, dO.at(off), dV.at(off), idS, kk > 0);
        }
        mma_commit_by(leader, &bars->v_empty[vs]);
        mma_commit_by(leader, &bars->sdp_full);
        if (c.i == c.n - 1) mma_commit_by(leader, &bars->qd_empty);
        return true;
      };
      auto next_a = [&](Cursor& c) {
        ++c.g;
        if (++c.i == c.n) {
          ++c.q;
          ++c.t;
          seek_a(c);
        }
      };
      Cursor A{0, 0, 0, 0, 0, 0, 0, 0, 0, false};
      seek_a(A);
      Cursor B = A;
      if (ok && !A.done) {
        if ((ok = issue_sdp(A))) next_a(A);
      }
      while (ok && !B.done) {
        // S / dP of the next block go first, unless that block starts another
        // item: then this row's last dQ goes first, so that the epilogue does
        // not wait behind the next row's MMAs (or its Q / dO loads); the next
        // S / dP run during the epilogue.
        const bool a_later = !A.done && A.i == 0;
        if (!A.done && !a_later) {
          if (!(ok = issue_sdp(A))) break;
          next_a(A);
          if (!ok) break;
        }
        const int st = B.g % C::kKStages;
        if (!(ok = warp_wait(&bars->ds_full[B.g & 1], (B.g >> 1) & 1, ab, a.status))) break;
        tc_fence_after();
        const SDesc dK(aK + st * C::kTile, 16384, 1024);
        const uint32_t ds = tmem + kColDS + (B.g & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_by(leader, tmem + kColDQ, ds + kk * 8, dK.at(kk * 2048), idDQ, (B.i > 0 || kk > 0) ? 1u : 0u);
        mma_commit_by(leader, &bars->k_empty[st]);
        mma_commit_by(leader, &bars->dq_done[B.g & 1]);
        __syncwarp();
        if (a_later) {
          if (!(ok = issue_sdp(A))) break;
          next_a(A);
          if (!ok) break;
        }
        ++B.g;
        if (++B.i == B.n) {
          __syncwarp();
          if (lane == 0) ring_release(ring, B.t);
          ++B.q;
          ++B.t;
          seek_b(B);
        }
      }
      mma_commit_by(leader, &bars->final_mma);
      if (leader) drain_wait(&bars->final_mma, 0);
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------- elementwise --
    const int hg = (warp - 2) / 4;  // column half
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const float sl2 = a.d.scale * kLog2e;
    int g = 0, sync_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int k = -1;
      if (lane == 0) ok = ring_get(ring, t, &k, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      k = __shfl_sync(0xffffffffu, k, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode_warp(k, cur);
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      T* dqrow = (T*)a.dQ + grow * D + hg * (D / 2);
      if (cur.n == 0) {
        zero_cols<D / 2>(dqrow);
      } else {
        const float lse2 = a.lse2[grow];
        const float dl = a.delta[grow];
        for (int i = 0; i < cur.n; ++i, ++g) {
          if (!(ok = warp_wait(&bars->sdp_full, g & 1, ab, a.status))) break;
          tc_fence_after();
          float s[64], dp[64];
          tmem_ld64(tmem + lane_base + kColS + hg * 64, s);
          tmem_ld64(tmem + lane_base + kColDP + hg * 64, dp);
          tc_fence_before();
          mbar_arrive(&bars->sdp_free);
          const float2 sc = make_float2(sl2, sl2), nl = make_float2(-lse2, -lse2), nd = make_float2(-dl, -dl);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float2 x = fma2(make_float2(s[2 * j], s[2 * j + 1]), sc, nl);
            const float2 y = mul2(make_float2(ex2(x.x), ex2(x.y)), add2(make_float2(dp[2 * j], dp[2 * j + 1]), nd));
            s[2 * j] = y.x;
            s[2 * j + 1] = y.y;
          }
          if (g > 1 && !(ok = warp_wait(&bars->dq_done[g & 1], ((g - 2) >> 1) & 1, ab, a.status))) break;
          tc_fence_after();
          tmem_st_pairs64<T>(tmem + lane_base + kColDS + (g & 1) * 64 + hg * 32, s);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->ds_full[g & 1]);
        }
        if (!ok) break;
        if (!(ok = warp_wait(&bars->dq_done[(g - 1) & 1], ((g - 1) >> 1) & 1, ab, a.status))) break;
        tc_fence_after();
        if (cur.slot < 0) {
          store_acc_cols<D / 2>(tmem + lane_base + kColDQ + hg * (D / 2), dqrow, a.d.scale, (size_t)D);
        } else {
          // chunk of a split row: publish the fp32 partial, the last chunk merges
          const size_t kTileF = (size_t)128 * D;
          store_acc_part<D / 2>(tmem + lane_base + kColDQ + hg * (D / 2),
                                a.part_q + (size_t)(cur.slot * a.d.BH + cur.bh) * kTileF, hg * (D / 8), r);
          bool last = false;
          if (!(ok = merge_arrive(lay, cur.slot, cur.bh, a.d.BH, hg, r, &bars->merge_flag[hg], &bars->wg_sync[hg],
                                  sync_phase, ab, a.status, &last)))
            break;
          if (last) {
            const int sl = lay.slot_line[cur.slot];
            const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
            merge_tiles<D / 2>(a.part_q + (size_t)(base * a.d.BH + cur.bh) * kTileF, (size_t)a.d.BH * kTileF, nc,
                               hg * (D / 8), r, dqrow, a.d.scale);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, t);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) plan_exit(lay);
}

// ================================================================ dK/dV ====
template <int D>
struct DkvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  // Q_g is read by S^T_g and, last, by dK_g; Q of block g+kQStages can only
  // load once dK_g is done, so Q gets one stage more than dO (read by dP^T_g
  // and dV_g, both early in the block).
  static constexpr int kQStages = D == 64 ? 4 : 3;
  static constexpr int kOStages = D == 64 ? 4 : 2;
  static constexpr int kStatStages = 2;
  static constexpr int kStat = 2 * 128 * 4;  // lse2 and delta of one block row's 128 queries
  static constexpr int kStatOff = kTile * (2 + kQStages + kOStages);
  static constexpr int kBarOff = kStatOff + kStatStages * kStat;
  // The dynamic shared memory base is 1024-byte aligned (checked at run
  // time), so this kernel, which needs almost all of the 227 KB, keeps no
  // alignment slack.
  static constexpr int kSmem = kBarOff + 512;
};

struct DkvBars {
  uint64_t k_full;
  uint64_t k_empty;  // the item's last S^T is done
  uint64_t v_full;
  uint64_t v_empty;  // the item's last dP^T is done
  uint64_t st_full;   // S^T of the block in TMEM
  uint64_t dpt_full;  // dP^T of the block in TMEM
  uint64_t pt_ready;  // P^T (over the S^T columns) in TMEM
  uint64_t ds_ready;  // dS^T (over the dP^T columns) in TMEM
  uint64_t pt_free;   // dV of the block done: the S^T columns are free
  uint64_t dk_done;   // dK of the block done: the dP^T columns are free
  uint64_t final_mma;
  uint64_t wg_sync[2];
  uint64_t stat_full[2];   // lse2 / delta of the block in shared memory
  uint64_t stat_empty[2];  // both warpgroups are done with them
  uint64_t q_full[4];
  uint64_t q_empty[4];
  uint64_t do_full[4];
  uint64_t do_empty[4];
  RingSmem ring;
  int merge_flag[2];
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(DkvBars) <= 512, "barrier block overflows its shared-memory slot");

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, BwdArgs a) {
  // may run as a programmatic dependent: the prologue below touches only
  // shared memory and TMEM; global memory waits for the previous grid
  griddep_launch_dependents();
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // no slack for re-alignment: refuse (uniform, before any barrier)
    griddep_wait();
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm;
  uint8_t* sV = sK + C::kTile;
  uint8_t* sQ = sV + C::kTile;
  uint8_t* sdO = sQ + C::kQStages * C::kTile;
  float* sStat = (float*)(sm + C::kStatOff);  // [stage][lse2 | delta][128]
  DkvBars* bars = (DkvBars*)(sm + C::kBarOff);
  // P^T (bf16) is written over the S^T columns and dS^T (bf16) over the dP^T
  // columns each warpgroup has read: queries [0, 64) at column +0, queries
  // [64, 128) at column +64.
  constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 256 + D;
  static_assert(kColDK + D <= kTmemCols, "TMEM columns over the allocation");
  static_assert(C::kSmem <= 232448, "shared memory over the per-CTA limit");

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const PlanLayout lay = plan_layout(a.col_plan, a.d.nb, (int)gridDim.x, a.d.BH);
  if (warp == 0) plan_prefetch_l2(a.col_plan, plan_words(a.d.nb, (int)gridDim.x, a.d.BH));

  if (threadIdx.x == 0) {
    mbar_init(&bars->k_full, 1);
    mbar_init(&bars->k_empty, 1);
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->dpt_full, 1);
    mbar_init(&bars->pt_ready, kEw);
    mbar_init(&bars->ds_ready, kEw);
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->wg_sync[i], 128);
      mbar_init(&bars->stat_full[i], 1);
      mbar_init(&bars->stat_empty[i], kEw);
    }
    for (int i = 0; i < C::kQStages; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < C::kOStages; ++i) {
      mbar_init(&bars->do_full[i], 1);
      mbar_init(&bars->do_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 1 + kEw / 32);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const Walk walk = make_walk(lay, a.d.BH);
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->ring;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      int g = 0, q = 0, vq = 0, lq = 0, ls = 0, lo = 0;  // blocks, items (K), V; Q / stats / dO loads issued
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        if (cur.n == 0) continue;
        // K of a new item once the previous item's last S^T is done; V
        // (first needed by dP^T) once its last dP^T is done, after the
        // first block's Q
        if (!(ok = mbar_wait(&bars->k_empty, (q & 1) ^ 1, ab, a.status))) break;
        const int krow = cur.bh * S + cur.line * 128;
        mbar_arrive_expect_tx(&bars->k_full, C::kTile);
        for (int b = 0; b < C::kBoxes; ++b) tma_load_2d(sK + b * 16384, &tmK, b * 64, krow, &bars->k_full);
        ++q;
        for (int i = 0; i < cur.n; ++i, ++g) {
          int m = a.row_idx[cur.first + i];
          if (m < 0 || m >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            m = 0;
          }
          const int qrow = cur.bh * S + m * 128;
          const int sq = g % C::kQStages, so = g % C::kOStages, ss = g % C::kStatStages;
          if (!(ok = mbar_wait(&bars->q_empty[sq], ((g / C::kQStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->q_full[sq], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sQ + sq * C::kTile + b * 16384, &tmQ, b * 64, qrow, &bars->q_full[sq]);
          lq = g + 1;
          if (!(ok = mbar_wait(&bars->stat_empty[ss], ((g / C::kStatStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->stat_full[ss], C::kStat);
          bulk_load(sStat + ss * 256, a.lse2 + qrow, 512, &bars->stat_full[ss]);
          bulk_load(sStat + ss * 256 + 128, a.delta + qrow, 512, &bars->stat_full[ss]);
          ls = g + 1;
          if (i == 0) {
            if (!(ok = mbar_wait(&bars->v_empty, (vq & 1) ^ 1, ab, a.status))) break;
            mbar_arrive_expect_tx(&bars->v_full, C::kTile);
            for (int b = 0; b < C::kBoxes; ++b) tma_load_2d(sV + b * 16384, &tmV, b * 64, krow, &bars->v_full);
            ++vq;
          }
          if (!(ok = mbar_wait(&bars->do_empty[so], ((g / C::kOStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->do_full[so], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sdO + so * C::kTile + b * 16384, &tmdO, b * 64, qrow, &bars->do_full[so]);
          lo = g + 1;
        }
      }
      // drain: every copy issued must land before the CTA exits
      if (q > 0) drain_wait(&bars->k_full, (q - 1) & 1);
      if (vq > 0) drain_wait(&bars->v_full, (vq - 1) & 1);
      for (int i = (lq > C::kQStages ? lq - C::kQStages : 0); i < lq; ++i)
        drain_wait(&bars->q_full[i % C::kQStages], (i / C::kQStages) & 1);
      for (int i = (ls > C::kStatStages ? ls - C::kStatStages : 0); i < ls; ++i)
        drain_wait(&bars->stat_full[i % C::kStatStages], (i / C::kStatStages) & 1);
      for (int i = (lo > C::kOStages ? lo - C::kOStages : 0); i < lo; ++i)
        drain_wait(&bars->do_full[i % C::kOStages], (i / C::kOStages) & 1);
    }
  } else if (warp == 1) {
    {
      // ----------------------------------------------------------- MMA --
      // The whole warp walks the schedule (descriptor arithmetic stays
      // warp-uniform); one elected lane issues the MMAs and commits.
      const uint32_t leader = elect_one();
      // Per block g the pipe runs dV_g, S^T_{g+1}, dK_g, dP^T_{g+1}:
      //   * dV_g (A = P^T from TMEM) as soon as P^T_g is there (pt_ready);
      //   * S^T_{g+1} overwrites P^T_g, so it waits for dV_g (pt_free);
      //   * dK_g (A = dS^T from TMEM) once dS^T_g is there (ds_ready);
      //   * dP^T_{g+1} overwrites dS^T_g, so it waits for dK_g (dk_done).
      // S^T_{g+1} is ready when the elementwise pass finishes block g; Q of
      // block g+3 loads as soon as dK_g is done.  When block g+1 starts
      // another item, dK_g goes before S^T_{g+1}, so that this item's
      // epilogue does not wait behind the next item's MMAs.
      const uint32_t idST = instr_desc(Half16<T>::kFmt, 0, 0, 128, 128);
      const uint32_t idG = instr_desc(Half16<T>::kFmt, 0, 1, D, 128);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), adO = smem_u32(sdO);
      bool ok = true;
      auto seek_a = [&](Cursor& c) {
        while (true) {
          int k;
          int kk0 = -1;
          bool good = true;
          if (lane == 0) good = ring_get(ring, c.t, &kk0, ab, a.status);
          ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
          k = __shfl_sync(0xffffffffu, kk0, 0);
          if (!ok || k < 0) {
            c.done = true;
            return;
          }
          walk.decode(k, c);
          if (c.n > 0) {
            c.i = 0;
            return;
          }
          ++c.t;
        }
      };
      auto seek_b = [&](Cursor& c) {
        while (true) {
          const int k = *(volatile int32_t*)&ring->k[c.t % kRing];
          if (k < 0) {
            c.done = true;
            return;
          }
          walk.decode(k, c);
          if (c.n > 0) {
            c.i = 0;
            return;
          }
          __syncwarp();
          if (lane == 0) ring_release(ring, c.t);
          ++c.t;
        }
      };
      auto next_a = [&](Cursor& c) {
        ++c.g;
        if (++c.i == c.n) {
          ++c.q;
          ++c.t;
          seek_a(c);
        }
      };
      auto issue_st = [&](const Cursor& c) -> bool {
        const int sq = c.g % C::kQStages;
        if (c.i == 0 && !warp_wait(&bars->k_full, c.q & 1, ab, a.status)) return false;
        if (!warp_wait(&bars->q_full[sq], (c.g / C::kQStages) & 1, ab, a.status)) return false;
        tc_fence_after();
        const SDesc dK(aK, 16, 1024), dQ(aQ + sq * C::kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_by(leader, tmem + kColST, dK.at(off), dQ.at(off), idST, kk > 0);
        }
        mma_commit_by(leader, &bars->st_full);
        if (c.i == c.n - 1) mma_commit_by(leader, &bars->k_empty);
        return true;
      };
      auto issue_dpt = [&](const Cursor& c) -> bool {
        const int so = c.g % C::kOStages;
        if (c.i == 0 && !warp_wait(&bars->v_full, c.q & 1, ab, a.status)) return false;
        if (!warp_wait(&bars->do_full[so], (c.g / C::kOStages) & 1, ab, a.status)) return false;
        tc_fence_after();
        const SDesc dV(aV, 16, 1024), dO(adO + so * C::kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_by(leader, tmem + kColDPT, dV.at(off), dO.at(off), idST, kk > 0);
        }
        mma_commit_by(leader, &bars->dpt_full);
        if (c.i == c.n - 1) mma_commit_by(leader, &bars->v_empty);
        return true;
      };
      Cursor A{0, 0, 0, 0, 0, 0, 0, 0, 0, false};
      seek_a(A);
      Cursor B = A;
      if (ok && !A.done) {
        if ((ok = issue_st(A) && issue_dpt(A))) next_a(A);
      }
      while (ok && !B.done) {
        const int sq = B.g % C::kQStages, so = B.g % C::kOStages;
        const SDesc dQmn(aQ + sq * C::kTile, 16384, 1024), dOmn(adO + so * C::kTile, 16384, 1024);
        if (!(ok = warp_wait(&bars->pt_ready, B.g & 1, ab, a.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_by(leader, tmem + kColDV, tmem + kColST + kk * 8 + (kk >= 4 ? 32 : 0), dOmn.at(kk * 2048), idG,
                         (B.i > 0 || kk > 0) ? 1u : 0u);
        mma_commit_by(leader, &bars->do_empty[so]);
        mma_commit_by(leader, &bars->pt_free);
        const bool a_first = !A.done && A.i == 0;  // the next block starts another item
        auto issue_s = [&]() -> bool {
          if (!warp_wait(&bars->pt_free, B.g & 1, ab, a.status)) return false;
          return issue_st(A);
        };
        if (!A.done && !a_first && !(ok = issue_s())) break;
        if (!(ok = warp_wait(&bars->ds_ready, B.g & 1, ab, a.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_by(leader, tmem + kColDK, tmem + kColDPT + kk * 8 + (kk >= 4 ? 32 : 0), dQmn.at(kk * 2048), idG,
                         (B.i > 0 || kk > 0) ? 1u : 0u);
        mma_commit_by(leader, &bars->q_empty[sq]);
        mma_commit_by(leader, &bars->dk_done);
        if (!A.done) {
          if (a_first && !(ok = issue_s())) break;
          if (!(ok = warp_wait(&bars->dk_done, B.g & 1, ab, a.status))) break;
          if (!(ok = issue_dpt(A))) break;
          next_a(A);
          if (!ok) break;
        }
        __syncwarp();
        ++B.g;
        if (++B.i == B.n) {
          __syncwarp();
          if (lane == 0) ring_release(ring, B.t);
          ++B.q;
          ++B.t;
          seek_b(B);
        }
      }
      mma_commit_by(leader, &bars->final_mma);
      if (leader) drain_wait(&bars->final_mma, 0);
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------- elementwise --
    const int hg = (warp - 2) / 4;  // query half of the tile
    const int wl = warp % 4;
    const int r = wl * 32 + lane;   // key row of the tile
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const float sl2 = a.d.scale * kLog2e;
    int g = 0, sync_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int k = -1;
      if (lane == 0) ok = ring_get(ring, t, &k, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      k = __shfl_sync(0xffffffffu, k, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode_warp(k, cur);
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      T* dkrow = (T*)a.dK + grow * D + hg * (D / 2);
      T* dvrow = (T*)a.dV + grow * D + hg * (D / 2);
      if (cur.n == 0) {
        zero_cols<D / 2>(dkrow);
        zero_cols<D / 2>(dvrow);
      } else {
        for (int i = 0; i < cur.n; ++i, ++g) {
          const int ss = g % C::kStatStages;
          int jb = -1;  // BSR position of the block, where its dS tile goes
          if (a.dS) {
            jb = a.bsr_of_bsc[cur.first + i];
            if (jb < 0 || jb >= a.nnzb) {
              atomicExch(a.status, kStatusDeviceCheck);
              jb = -1;
            }
          }
          if (!(ok = warp_wait(&bars->st_full, g & 1, ab, a.status))) break;
          if (!(ok = warp_wait(&bars->stat_full[ss], (g / C::kStatStages) & 1, ab, a.status))) break;
          tc_fence_after();
          float s[64], dp[64];
          tmem_ld64(tmem + lane_base + kColST + hg * 64, s);
          // statistics of this block row's queries (bulk-copied by the producer)
          const float* lse = sStat + ss * 256 + hg * 64;
          const float* dl = lse + 128;
          const float2 sc = make_float2(sl2, sl2);
          // (statistics four at a time: the ring's stage is 16-byte aligned)
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 l4 = *(const float4*)(lse + 4 * k);
            const float2 x = fma2(make_float2(s[4 * k], s[4 * k + 1]), sc, make_float2(-l4.x, -l4.y));
            const float2 y = fma2(make_float2(s[4 * k + 2], s[4 * k + 3]), sc, make_float2(-l4.z, -l4.w));
            s[4 * k] = ex2(x.x);
            s[4 * k + 1] = ex2(x.y);
            s[4 * k + 2] = ex2(y.x);
            s[4 * k + 3] = ex2(y.y);
          }
          // P^T over this warpgroup's own S^T columns (already read above;
          // dV of the previous block finished before S^T of this one began)
          tmem_st_pairs64<T>(tmem + lane_base + kColST + hg * 64, s);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->pt_ready);
          if (!(ok = warp_wait(&bars->dpt_full, g & 1, ab, a.status))) break;
          tc_fence_after();
          tmem_ld64(tmem + lane_base + kColDPT + hg * 64, dp);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 d4 = *(const float4*)(dl + 4 * k);
            const float2 x = mul2(make_float2(s[4 * k], s[4 * k + 1]),
                                  add2(make_float2(dp[4 * k], dp[4 * k + 1]), make_float2(-d4.x, -d4.y)));
            const float2 y = mul2(make_float2(s[4 * k + 2], s[4 * k + 3]),
                                  add2(make_float2(dp[4 * k + 2], dp[4 * k + 3]), make_float2(-d4.z, -d4.w)));
            dp[4 * k] = x.x;
            dp[4 * k + 1] = x.y;
            dp[4 * k + 2] = y.x;
            dp[4 * k + 3] = y.y;
          }
          mbar_arrive(&bars->stat_empty[ss]);
          // dS^T over this warpgroup's own dP^T columns (read above; dK of
          // the previous block finished before dP^T of this one began)
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = Half16<T>::pack(dp[2 * k], dp[2 * k + 1]);
          tmem_st32(tmem + lane_base + kColDPT + hg * 64, w);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->ds_ready);
          if (jb >= 0)  // the dS tile of (block row m, this column), in the layout dq_ds_kernel stages
            st_tile_sw32_row64((uint8_t*)a.dS + ((size_t)cur.bh * a.nnzb + jb) * (128 * 128 * 2), r, hg, w);
        }
        if (!ok) break;
        if (cur.slot < 0) {
          // dV is final once the item's last dV is done (pt_free), while its
          // last dK may still run
          if (!(ok = warp_wait(&bars->pt_free, (g - 1) & 1, ab, a.status))) break;
          tc_fence_after();
          store_acc_cols<D / 2>(tmem + lane_base + kColDV + hg * (D / 2), dvrow, 1.f, (size_t)D);
          if (!(ok = warp_wait(&bars->dk_done, (g - 1) & 1, ab, a.status))) break;
          tc_fence_after();
          store_acc_cols<D / 2>(tmem + lane_base + kColDK + hg * (D / 2), dkrow, a.d.scale, (size_t)D);
        } else {
          if (!(ok = warp_wait(&bars->dk_done, (g - 1) & 1, ab, a.status))) break;
          tc_fence_after();
          // chunk of a split column: publish the fp32 partials, the last chunk merges
          const size_t kTileF = (size_t)128 * D;
          const size_t tile = (size_t)cur.slot * a.d.BH + cur.bh;
          store_acc_part<D / 2>(tmem + lane_base + kColDV + hg * (D / 2), a.part_kv + (tile * 2 + 0) * kTileF,
                                hg * (D / 8), r);
          store_acc_part<D / 2>(tmem + lane_base + kColDK + hg * (D / 2), a.part_kv + (tile * 2 + 1) * kTileF,
                                hg * (D / 8), r);
          bool last = false;
          if (!(ok = merge_arrive(lay, cur.slot, cur.bh, a.d.BH, hg, r, &bars->merge_flag[hg], &bars->wg_sync[hg],
                                  sync_phase, ab, a.status, &last)))
            break;
          if (last) {
            const int sl = lay.slot_line[cur.slot];
            const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
            const size_t t0 = (size_t)base * a.d.BH + cur.bh;
            const size_t stride = (size_t)a.d.BH * 2 * kTileF;  // next slot, same head
            merge_tiles<D / 2>(a.part_kv + (t0 * 2 + 0) * kTileF, stride, nc, hg * (D / 8), r, dvrow, 1.f);
            merge_tiles<D / 2>(a.part_kv + (t0 * 2 + 1) * kTileF, stride, nc, hg * (D / 8), r, dkrow, a.d.scale);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, t);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) plan_exit(lay);
}

// ========================================================== dQ from dS ====
// On a plan the dK/dV walk stores each dS tile it computes (a.dS), and the
// dQ walk becomes dQ_m = scale * sum_n dS_mn K_n over them: one MMA group
// per stored block, no recomputed scores, no statistics.  It still walks
// block rows with one writer per dQ tile ("trnsparse 0.4.1 -> 0.6.0" diff,
// CHANGELOG [0.5.1]); what it saves is the S and dP products (two of the
// three MMA groups of the recomputing walk) for 32 KB of dS written and read
// back per block, which HBM has room for beside the MMA-bound dK/dV walk.
//
// A dS tile (128 queries x 128 keys, 16-bit) sits in memory as the dK/dV
// walk writes it: the MN-major operand layout with 32-byte swizzling, so a
// plain bulk copy to a 1024-byte aligned stage is ready for the MMA as the
// A operand of dQ += dS K (M = queries, K = keys).  Its atoms are 8 keys x
// 16 queries (8 rows of 32 bytes, the 16-byte halves of rows 4..7 swapped);
// the atoms of the next 8 keys follow at 256 bytes (stride byte offset) and
// those of the next 16 queries at 4096 bytes (leading byte offset).
//
// A work item covers W = min(D, 256) output columns: head_dim 512 runs as
// two slices, planned as heads of their own (the wide kernels' plan, so a
// split row's chunks merge per slice), each reading every dS tile of its row
// once and the slice's columns of K.
//
// Warp roles (320 threads): warp 0 the producer (the tile pair of each block
// through a ring of stages), warp 1 TMEM owner and MMA issuer, warps 2..9
// the epilogue (thread (w, l) owns dQ row 32 (w % 4) + l and half of the
// slice's columns), which stores an item's dQ from one of two TMEM
// accumulators while the MMAs of the next item fill the other.
template <int D>
struct DsCfg {
  static constexpr int W = D < 256 ? D : 256;  // output columns per work item
  static constexpr int NSL = D / W;
  static constexpr int kBoxes = W / 64;
  static constexpr int kKTile = 128 * W * 2;
  static constexpr int kDsTile = 128 * 128 * 2;
  static constexpr int kStageBytes = kDsTile + kKTile;  // a multiple of 1024 (the K boxes are swizzled)
  static constexpr int kStages = D == 64 ? 4 : (W == 256 ? 2 : 3);
  static constexpr int kBarOff = kStageBytes * kStages;
  static constexpr int kSmem = kBarOff + 512 + 1024;
  static constexpr uint32_t kCols = 2 * W <= 128 ? 128 : (2 * W <= 256 ? 256 : 512);  // two accumulators of W columns
};

struct DsBars {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t acc_full[2];   // the item's last MMA into accumulator b is done
  uint64_t acc_empty[2];  // the epilogue has read accumulator b
  uint64_t final_mma;
  uint64_t wg_sync[2];
  RingSmem ring;
  int merge_flag[2];
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(DsBars) <= 512, "barrier block overflows its shared-memory slot");

// kDV: the same streaming walk for dV at head_dim 256 / 512 on a plan: the
// wide dK walk also stores each P^T tile (keys x queries, in BSC order, the
// same byte layout: read here as the K-major A operand with 32-byte
// swizzling, M = keys: 8 keys x 16 queries per atom, the next 8 keys 256
// bytes on, the next 16 queries 4096 bytes on), and dV_n = sum_m P^T_nm dO_m
// walks the block columns (the dV plan, dO as the B operand, no scale).
template <typename T, int D, bool kDV>
__global__ void __launch_bounds__(kThreads, 1) dq_ds_kernel(const __grid_constant__ CUtensorMap tmK, BwdArgs a) {
  // runs as a programmatic dependent of the dK/dV walk: the prologue below
  // touches only shared memory and TMEM; global memory waits for that grid
  griddep_launch_dependents();
  using C = DsCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  DsBars* bars = (DsBars*)(sm + C::kBarOff);
  static_assert(C::kSmem <= 232448, "shared memory over the per-CTA limit");
  static_assert(C::kStageBytes % 1024 == 0, "stages must keep the 1024-byte alignment of the swizzled boxes");

  constexpr int W = C::W, NSL = C::NSL;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const int BHp = a.d.BH * NSL;  // the planner's heads: one per (batch, head, slice)
  int32_t* const plan = kDV ? a.col_plan : a.row_plan;
  const int32_t* const idx = kDV ? a.row_idx : a.col_idx;
  const uint8_t* const tiles = (const uint8_t*)(kDV ? a.dP : a.dS);
  T* const out = (T*)(kDV ? a.dV : a.dQ);
  float* const part = kDV ? a.part_kv : a.part_q;
  const float mul = kDV ? 1.f : a.d.scale;
  const PlanLayout lay = plan_layout(plan, a.d.nb, (int)gridDim.x, BHp);
  if (warp == 0) plan_prefetch_l2(plan, plan_words(a.d.nb, (int)gridDim.x, BHp));

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], kEw);
      mbar_init(&bars->wg_sync[i], 128);
    }
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 1 + kEw / 32);  // MMA warp + epilogue warps
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, C::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const Walk walk = make_walk(lay, BHp);
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->ring;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      int g = 0;  // blocks whose copies were issued
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        const int bh = cur.bh / NSL, sl = cur.bh % NSL;
        // the line's tiles are consecutive (dS: BSR order; P^T: BSC order)
        const uint8_t* ds = tiles + ((size_t)bh * a.nnzb + cur.first) * C::kDsTile;
        for (int i = 0; i < cur.n; ++i, ++g) {
          int n = idx[cur.first + i];
          if (n < 0 || n >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            n = 0;
          }
          const int st = g % C::kStages;
          if (!(ok = mbar_wait(&bars->empty[st], ((g / C::kStages) & 1) ^ 1, ab, a.status))) break;
          uint8_t* dst = sm + st * C::kStageBytes;
          mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
          bulk_load(dst, ds + (size_t)i * C::kDsTile, C::kDsTile / 2, &bars->full[st]);
          bulk_load(dst + C::kDsTile / 2, ds + (size_t)i * C::kDsTile + C::kDsTile / 2, C::kDsTile / 2,
                    &bars->full[st]);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(dst + C::kDsTile + b * 16384, &tmK, sl * W + b * 64, bh * S + n * 128, &bars->full[st]);
        }
      }
      // drain: every copy issued must land before the CTA exits
      for (int i = (g > C::kStages ? g - C::kStages : 0); i < g; ++i)
        drain_wait(&bars->full[i % C::kStages], (i / C::kStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA --
    const uint32_t leader = elect_one();
    const uint32_t idDQ = instr_desc(Half16<T>::kFmt, kDV ? 0 : 1, 1, W, 128);
    const uint32_t base = smem_u32(sm);
    int g = 0, q = 0;  // blocks, non-empty items
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int k0 = -1;
      bool good = true;
      if (lane == 0) good = ring_get(ring, t, &k0, ab, a.status);
      ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
      const int k = __shfl_sync(0xffffffffu, k0, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode(k, cur);
      if (cur.n > 0) {
        const int buf = q & 1;
        if (!(ok = warp_wait(&bars->acc_empty[buf], ((q >> 1) & 1) ^ 1, ab, a.status))) break;
        tc_fence_after();
        for (int i = 0; i < cur.n; ++i, ++g) {
          const int st = g % C::kStages;
          if (!(ok = warp_wait(&bars->full[st], (g / C::kStages) & 1, ab, a.status))) break;
          tc_fence_after();
          const uint32_t sds = base + st * C::kStageBytes;
          // dS: MN-major with 32-byte swizzle; P^T (kDV): K-major with 32-byte
          // swizzle (one atom per MMA's 16 queries: the leading offset is unused)
          const uint64_t dA = kDV ? smem_desc(sds, 16, 256, 6) : smem_desc(sds, 4096, 256, 6);
          const SDesc dK(sds + C::kDsTile, 16384, 1024);  // K / dO: MN-major, 128-byte swizzle
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // 16 keys (queries for kDV) per MMA: 16 rows of K (dO)
            mma_ss_by(leader, tmem + buf * W, dA + (uint64_t)(kk * (kDV ? 256 : 32)), dK.at(kk * 2048), idDQ,
                      (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit_by(leader, &bars->empty[st]);
        }
        if (!ok) break;
        mma_commit_by(leader, &bars->acc_full[buf]);
        ++q;
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, t);
    }
    mma_commit_by(leader, &bars->final_mma);
    if (leader) drain_wait(&bars->final_mma, 0);
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue --
    const int hg = (warp - 2) / 4;  // column half
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    int q = 0, sync_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int k = -1;
      if (lane == 0) ok = ring_get(ring, t, &k, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      k = __shfl_sync(0xffffffffu, k, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode_warp(k, cur);
      const int bh = cur.bh / NSL, sl = cur.bh % NSL;
      const size_t grow = (size_t)bh * S + (size_t)cur.line * 128 + r;
      T* dqrow = out + grow * D + sl * W + hg * (W / 2);
      if (cur.n == 0) {
        zero_cols<W / 2>(dqrow);
      } else {
        const int buf = q & 1;
        if (!(ok = warp_wait(&bars->acc_full[buf], (q >> 1) & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t acc = tmem + lane_base + buf * W + hg * (W / 2);
        ++q;
        if (cur.slot < 0) {
          store_acc_cols<W / 2>(acc, dqrow, mul, (size_t)D);
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[buf]);
        } else {
          // chunk of a split row: publish the fp32 partial, the last chunk merges
          const size_t kTileF = (size_t)128 * W;
          store_acc_part<W / 2>(acc, part + (size_t)(cur.slot * BHp + cur.bh) * kTileF, hg * (W / 8), r);
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[buf]);
          bool last = false;
          if (!(ok = merge_arrive(lay, cur.slot, cur.bh, BHp, hg, r, &bars->merge_flag[hg], &bars->wg_sync[hg],
                                  sync_phase, ab, a.status, &last)))
            break;
          if (last) {
            const int sl = lay.slot_line[cur.slot];
            const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
            merge_tiles<W / 2>(part + (size_t)(base * BHp + cur.bh) * kTileF, (size_t)BHp * kTileF, nc,
                               hg * (W / 8), r, dqrow, mul);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, t);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kCols);
  if (threadIdx.x == 0) plan_exit(lay);
}

// The dQ walk over the stored dS tiles, in `s` as a programmatic dependent
// of the walk that stored them.
template <typename T, int D, bool kDV = false>
bsr_status launch_dq(const BwdArgs& a, const CUtensorMap& tmB, int grid, cudaStream_t s) {
  auto dq = dq_ds_kernel<T, D, kDV>;
  const char* name = kDV ? "dv_ps" : "dq_ds";
  cudaError_t e = cudaFuncSetAttribute(dq, cudaFuncAttributeMaxDynamicSharedMemorySize, DsCfg<D>::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "%s: cudaFuncSetAttribute(%d): %s", name, DsCfg<D>::kSmem, cudaGetErrorString(e));
  if (profiling_launches()) {
    LaunchTimer timer(name, s);
    dq<<<grid, kThreads, DsCfg<D>::kSmem, s>>>(tmB, a);
    return check_launch(name);
  }
  e = launch_dependent(dq, dim3(grid), dim3(kThreads), DsCfg<D>::kSmem, s, tmB, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

// On a plan (a.dS set): the dK/dV walk, which stores the dS tiles, then the
// dQ walk over them, both in `s` as programmatic dependents.
template <typename T, int D>
bsr_status launch_bwd_ds(const BwdArgs& a, const TensorMaps& tm, const CUtensorMap& tmdO, int grid, cudaStream_t s) {
  auto dkdv = dkdv_tc_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvCfg<D>::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "dkdv_tc: cudaFuncSetAttribute(%d): %s", DkvCfg<D>::kSmem, cudaGetErrorString(e));
  if (profiling_launches()) {
    LaunchTimer timer("dkdv_tc", s);
    dkdv<<<grid, kThreads, DkvCfg<D>::kSmem, s>>>(tm.q, tm.k, tm.v, tmdO, a);
    bsr_status st = check_launch("dkdv_tc launch");
    if (st != BSR_OK) return st;
  } else {
    e = launch_dependent(dkdv, dim3(grid), dim3(kThreads), DkvCfg<D>::kSmem, s, tm.q, tm.k, tm.v, tmdO, a);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "dkdv_tc launch: %s", cudaGetErrorString(e));
    bsr_status st = check_launch("dkdv_tc launch");
    if (st != BSR_OK) return st;
  }
  return launch_dq<T, D>(a, tm.k, grid, s);
}

// dQ and dK / dV read the same inputs and write different outputs, so they
// run side by side: dK / dV on a second stream forked from `s` and joined
// back into it.  Their CTAs never share an SM (each needs almost all of its
// shared memory), so the second kernel's CTAs take the SMs the first one
// leaves in its tail.
template <typename T, int D>
bsr_status launch_bwd(const BwdArgs& a, const TensorMaps& tm, const CUtensorMap& tmdO, int grid, cudaStream_t s) {
  auto dq = dq_tc_kernel<T, D>;
  auto dkdv = dkdv_tc_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(dq, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "dq_tc: cudaFuncSetAttribute(%d): %s", DqCfg<D>::kSmem, cudaGetErrorString(e));
  e = cudaFuncSetAttribute(dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvCfg<D>::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "dkdv_tc: cudaFuncSetAttribute(%d): %s", DkvCfg<D>::kSmem, cudaGetErrorString(e));
  if (profiling_launches()) {  // one after the other, each timed alone
    {
      LaunchTimer timer("dq_tc", s);
      dq<<<grid, kThreads, DqCfg<D>::kSmem, s>>>(tm.q, tm.k, tm.v, tmdO, a);
      bsr_status st = check_launch("dq_tc launch");
      if (st != BSR_OK) return st;
    }
    LaunchTimer timer("dkdv_tc", s);
    dkdv<<<grid, kThreads, DkvCfg<D>::kSmem, s>>>(tm.q, tm.k, tm.v, tmdO, a);
    return check_launch("dkdv_tc launch");
  }
  SideStream side;
  std::unique_lock<std::mutex> hold;
  bsr_status st = side_stream(&side, &hold);
  if (st != BSR_OK) return st;
  if ((e = cudaEventRecord(side.fork, s)) != cudaSuccess || (e = cudaStreamWaitEvent(side.s, side.fork, 0)) != cudaSuccess)
    return fail(BSR_ERR_CUDA, "bwd_tc: fork: %s", cudaGetErrorString(e));
  dkdv<<<grid, kThreads, DkvCfg<D>::kSmem, side.s>>>(tm.q, tm.k, tm.v, tmdO, a);
  st = check_launch("dkdv_tc launch");
  if (st == BSR_OK) {
    e = launch_dependent(dq, dim3(grid), dim3(kThreads), DqCfg<D>::kSmem, s, tm.q, tm.k, tm.v, tmdO, a);
    st = e != cudaSuccess ? fail(BSR_ERR_CUDA, "dq_tc launch: %s", cudaGetErrorString(e)) : check_launch("dq_tc launch");
  }
  // join even after a failed launch, so `s` stays ordered after the side stream
  if ((e = cudaEventRecord(side.join, side.s)) != cudaSuccess || (e = cudaStreamWaitEvent(s, side.join, 0)) != cudaSuccess)
    return fail(BSR_ERR_CUDA, "bwd_tc: join: %s", cudaGetErrorString(e));
  return st;
}

}  // namespace

bsr_status launch_dq_ds(const BwdArgs& a, cudaStream_t s) {
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "dq_ds: cannot query the SM count");
  if (!a.dS || (((uintptr_t)a.dS) & 15) || a.d.dtype == BSR_F32)
    return fail(BSR_ERR_INVALID_ARG, "dq_ds: needs 16-byte aligned dS tiles of 16-bit operands");
  CUtensorMap tmK;
  bsr_status st = make_tensor_map(a.d, a.K, &tmK, "K");
  if (st != BSR_OK) return st;
  const bool h = a.d.dtype == BSR_F16;
  switch (a.d.D) {
    case 256: return h ? launch_dq<__half, 256>(a, tmK, grid, s) : launch_dq<__nv_bfloat16, 256>(a, tmK, grid, s);
    case 512: return h ? launch_dq<__half, 512>(a, tmK, grid, s) : launch_dq<__nv_bfloat16, 512>(a, tmK, grid, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "dq_ds: head_dim %d", a.d.D);
  }
}

bsr_status launch_dv_ps(const BwdArgs& a, cudaStream_t s) {
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "dv_ps: cannot query the SM count");
  if (!a.dP || (((uintptr_t)a.dP) & 15) || a.d.dtype == BSR_F32)
    return fail(BSR_ERR_INVALID_ARG, "dv_ps: needs 16-byte aligned P^T tiles of 16-bit operands");
  CUtensorMap tmdO;
  bsr_status st = make_tensor_map(a.d, a.dO, &tmdO, "dO");
  if (st != BSR_OK) return st;
  const bool h = a.d.dtype == BSR_F16;
  switch (a.d.D) {
    case 256:
      return h ? launch_dq<__half, 256, true>(a, tmdO, grid, s) : launch_dq<__nv_bfloat16, 256, true>(a, tmdO, grid, s);
    case 512:
      return h ? launch_dq<__half, 512, true>(a, tmdO, grid, s) : launch_dq<__nv_bfloat16, 512, true>(a, tmdO, grid, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "dv_ps: head_dim %d", a.d.D);
  }
}

bool tc_bwd_supported(const Dims& d) {
  return (d.dtype == BSR_BF16 || d.dtype == BSR_F16) && (d.D == 64 || d.D == 128);
}

int tc_grid(const Dims& d) {
  const int sms = sm_count();
  const int total = d.nb * d.BH;
  return sms <= 0 ? 0 : (total < sms ? total : sms);
}

bsr_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
  if ((((uintptr_t)a.lse2) | ((uintptr_t)a.delta)) & 15)
    return fail(BSR_ERR_INVALID_ARG, "bwd_tc: scratch arrays must be 16-byte aligned");
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "bwd_tc: cannot query the SM count");
  TensorMaps tm;
  bsr_status st = make_tensor_maps(a.d, a.Q, a.K, a.V, &tm);
  if (st != BSR_OK) return st;
  CUtensorMap tmdO;
  if ((st = make_tensor_map(a.d, a.dO, &tmdO, "dO")) != BSR_OK) return st;
  if (a.dS && (((uintptr_t)a.dS) & 15 || !a.bsr_of_bsc))
    return fail(BSR_ERR_INVALID_ARG, "bwd_tc: the dS tiles need 16-byte alignment and the BSC-to-BSR map");
  const bool ds = a.dS != nullptr;
  switch (a.d.D) {
    case 64:
      if (ds)
        return a.d.dtype == BSR_F16 ? launch_bwd_ds<__half, 64>(a, tm, tmdO, grid, s)
                                    : launch_bwd_ds<__nv_bfloat16, 64>(a, tm, tmdO, grid, s);
      return a.d.dtype == BSR_F16 ? launch_bwd<__half, 64>(a, tm, tmdO, grid, s)
                                  : launch_bwd<__nv_bfloat16, 64>(a, tm, tmdO, grid, s);
    case 128:
      if (ds)
        return a.d.dtype == BSR_F16 ? launch_bwd_ds<__half, 128>(a, tm, tmdO, grid, s)
                                    : launch_bwd_ds<__nv_bfloat16, 128>(a, tm, tmdO, grid, s);
      return a.d.dtype == BSR_F16 ? launch_bwd<__half, 128>(a, tm, tmdO, grid, s)
                                  : launch_bwd<__nv_bfloat16, 128>(a, tm, tmdO, grid, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "bwd_tc: head_dim %d", a.d.D);
  }
}

}  // namespace bsr
