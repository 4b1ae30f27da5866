// Tensor-core forward pass for 16-bit operands (bf16 or fp16, fp32
// accumulation) with head_dim 64 / 128 on sm_103a, with P kept in tensor
// memory in the operand type.
//
// For each block row m of one (batch, head) the row's stored blocks j in
// [row_ptr[m], row_ptr[m+1]) are visited in order and the K / V tiles of
// block column col_idx[j] come straight from HBM by TMA ("trnsparse 0.7.0 ->
// 0.9.0" diff, CHANGELOG [0.8.0], attn_fwd_static: one launch, statistics on
// chip, no K/V gather, no per-block score round trip through HBM), with
// these choices that keep the tensor pipe fed:
//   * persistent CTAs, one per SM, take (row, head) work items longest row
//     first from a queue (sched.cuh) and prefetch the next item's Q (two Q
//     buffers) and K / V tiles while the current one finishes;
//   * the 128 keys of every block are split into two halves of 64, and each
//     half has its own softmax warpgroup with its own online-softmax state
//     (running reference max, row sum) and its own O accumulator
//     O_h = sum_j P_hj V_hj.  The halves never talk to each other inside a
//     row; once per row the two partial results are combined exactly like
//     two chunks of a split row:  R = max(m_0, m_1),
//     O = (2^(m_0 - R) O_0 + 2^(m_1 - R) O_1) / (2^(m_0 - R) l_0 + 2^(m_1 - R) l_1);
//   * P goes back to tensor memory in the operand type (two buffers) and
//     the P.V MMA reads its A operand from there;
//   * S has one TMEM buffer, released as soon as both warpgroups have
//     loaded their halves into registers, so S_{j+1} = Q K_{j+1}^T runs
//     while the softmax of block j is computed;
//   * two threads issue the MMAs, one the S and one the P.V of every block,
//     each as soon as its operands are there (issue and commit cost a
//     thread tens to a hundred cycles each, and each MMA thread waits on
//     barriers that the other one does not need);
//   * the producer keeps the work ring one item ahead of the item it loads,
//     so the global work counter's round trip is off the item boundary.
// The same kernel also runs the two launches of the statistics-first
// variant (kStatsPass, kOutPass below).
//
// Warp roles (384 threads): warp 0 TMA producer of Q and K, warp 10 TMA
// producer of V, warp 1 TMEM owner and issuer of the S MMAs, warp 11 issuer
// of the P.V MMAs, warps 2..9 two softmax warpgroups; thread (warp w, lane
// l) owns query row 32 (w % 4) + l (its TMEM lane), warpgroup
// h = (w - 2) / 4 owns keys [64 h, 64 h + 64) of each block and, in the
// final combine, output columns [h D / 2, h D / 2 + D / 2).
// TMEM columns: S at 0 (half h at +64 h), P of block j at 128 + 64 (j % 2)
// (half h at +32 h), O_0 at 256, O_1 at 256 + D.  All waits are bounded
// (see sm100.cuh).

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

constexpr int kThreads = 384;  // producer, S MMAs, 8 softmax warps, V producer, P.V MMAs
constexpr int kWarpV = 10;
constexpr int kWarpPV = 11;
constexpr int kSoftmax = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 128, kColO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max may lag by 2^8

// Forward variants: the single online-softmax pass, or the two launches of
// the statistics-first variant ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG
// [0.4.3]: the row statistics in a first pass over the row's blocks, the
// output in a second one with P normalised by them).  The statistics pass
// issues no P.V and loads no V; the output pass takes no maximum and never
// rescales.
constexpr int kOnline = 0, kStatsPass = 1, kOutPass = 2;

template <int D>
struct Fwd2Cfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kQStages = 2;
  static constexpr int kKStages = D == 64 ? 4 : 3;
  static constexpr int kVStages = D == 64 ? 4 : 2;
  static constexpr int kRedOff = kTile * (kQStages + kKStages + kVStages);
  // per row: m_ref_0, l_0, m_ref_1, l_1, m_true_1 (the row statistics are
  // written by warpgroup 0, which needs the other half's true maximum)
  static constexpr int kRedFloats = 5 * 128;
  static constexpr int kBarOff = kRedOff + kRedFloats * 4;
  // The dynamic shared memory base is 1024-byte aligned (checked at run
  // time); with head_dim 128 the tiles take almost all of the 227 KB, so no
  // alignment slack is kept.
  static constexpr int kSmem = kBarOff + 512;
  static_assert(kSmem <= 232448, "shared memory over the per-CTA limit");
  // TMEM: S (128 columns), two P buffers of 64, O_0 and O_1 (D each)
  static_assert(kColP + 2 * 64 <= kColO && kColO + 2 * D <= kTmemCols, "TMEM columns over the allocation");
};

struct Bars {
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full;
  uint64_t s_free;      // both warpgroups have loaded S into registers
  uint64_t p_full[2];     // by P buffer b: both halves' P of block g (g % 2 = b) are in TMEM
  uint64_t pv_done[2];    // by P buffer b: both halves' P.V of block g (g % 2 = b) are done
  uint64_t final_mma[2];  // by MMA thread (S, P.V): all its MMAs are done
  uint64_t red_full;   // both warpgroups' row statistics written
  uint64_t red_empty;  // both warpgroups have read them
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
static_assert(sizeof(Bars) <= 512, "barrier block overflows its shared-memory slot");

// Partial result of one chunk of a split row (fp32): O (128 x D, relative to
// the chunk's reference max) then, per column half and row, the chunk's
// reference max, row sum and an upper bound of the row's maximum (the true
// maximum in half 0, whose merge writes the row statistics; log2 units) and
// a pad.
template <int D>
__host__ __device__ constexpr size_t fwd_part_floats() {
  return (size_t)128 * D + 2 * 128 * 4;
}

// Largest (or, for a negative scale, smallest) of 64 raw scores: eight
// chains of three-input max, then a tree.
template <bool kMax>
__device__ __forceinline__ float extreme64(const float (&v)[64]) {
  float c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float* x = v + 8 * j;
    if (kMax) {
      c[j] = max3f(max3f(max3f(x[0], x[1], x[2]), x[3], x[4]), x[5], x[6]);
      c[j] = fmaxf(c[j], x[7]);
    } else {
      c[j] = min3f(min3f(min3f(x[0], x[1], x[2]), x[3], x[4]), x[5], x[6]);
      c[j] = fminf(c[j], x[7]);
    }
  }
  if (kMax) return max3f(max3f(c[0], c[1], c[2]), max3f(c[3], c[4], c[5]), fmaxf(c[6], c[7]));
  return min3f(min3f(c[0], c[1], c[2]), min3f(c[3], c[4], c[5]), fminf(c[6], c[7]));
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Bars* b, int* status) {
  bool ok = mbar_wait(bar, parity, &b->abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

template <typename T, int D, int kPass>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  // may run as a programmatic dependent: the prologue below touches only
  // shared memory and TMEM; global memory waits for the previous grid
  griddep_launch_dependents();
  using C = Fwd2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // no slack for re-alignment: refuse (uniform, before any barrier)
    griddep_wait();
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + C::kQStages * C::kTile;
  uint8_t* sV = sK + C::kKStages * C::kTile;
  float* sRed = (float*)(sm + C::kRedOff);
  Bars* bars = (Bars*)(sm + C::kBarOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const PlanLayout lay = plan_layout(a.plan, a.d.nb, (int)gridDim.x, a.d.BH);
  if (warp == 0) plan_prefetch_l2(a.plan, plan_words(a.d.nb, (int)gridDim.x, a.d.BH));

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->p_full[i], kSoftmax);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->wg_sync[i], 128);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, kSoftmax);
    mbar_init(&bars->final_mma[0], 1);
    mbar_init(&bars->final_mma[1], 1);
    mbar_init(&bars->red_full, kSoftmax);
    mbar_init(&bars->red_empty, kSoftmax);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 3 + kSoftmax / 32);  // two MMA threads, softmax warps, V producer
    }
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
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
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int kg = 0, q = 0, g = 0;
      int put = 0;         // ring slots published
      bool ended = false;  // the slot that ends the walk is published
      bool ok = true;
      auto publish = [&](int upto) -> bool {  // ring slots [put, upto)
        for (; put < upto && !ended; ++put) {
          int kk;
          if (!ring_put(ring, put, lay.header + 1, walk.total, &kk, ab, a.status)) return false;
          ended = kk < 0;
        }
        return true;
      };
      for (int t = 0; ok; ++t) {
        if (!(ok = publish(t + 1))) break;
        const int k = *(volatile int32_t*)&ring->k[t % kRing];
        if (k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        if (cur.n == 0) continue;
        // Q of item q goes to buffer q % 2 once item q - 2's S MMAs are done
        const int qb = q & 1;
        if (!(ok = mbar_wait(&bars->q_empty[qb], ((q >> 1) & 1) ^ 1, ab, a.status))) break;
        const int qrow = cur.bh * S + cur.line * 128;
        mbar_arrive_expect_tx(&bars->q_full[qb], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sQ + qb * C::kTile + b * 16384, &tmQ, b * 64, qrow, &bars->q_full[qb]);
        ++q;
        // the next item's slot (and the work counter's round trip) while
        // this item's K tiles load
        if (!(ok = publish(t + 2))) break;
        for (int j = 0; j < cur.n; ++j, ++g) {
          int n = a.col_idx[cur.first + j];
          if (n < 0 || n >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            n = 0;
          }
          const int krow = cur.bh * S + n * 128;
          const int ks = g % C::kKStages;
          if (!(ok = mbar_wait(&bars->k_empty[ks], ((g / C::kKStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->k_full[ks], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sK + ks * C::kTile + b * 16384, &tmK, b * 64, krow, &bars->k_full[ks]);
          kg = g + 1;
        }
      }
      // drain: every copy issued must have landed before the CTA exits
      for (int i = (q > 2 ? q - 2 : 0); i < q; ++i) drain_wait(&bars->q_full[i & 1], (i >> 1) & 1);
      for (int i = (kg > C::kKStages ? kg - C::kKStages : 0); i < kg; ++i)
        drain_wait(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1);
    }
  } else if (warp == kWarpV) {
    if (lane == 0) {
      // ---------------------------------------------------- V producer --
      // V runs on its own thread so that K (needed first, by S) is never
      // held back behind a V stage that is still in use by P.V.
      int vg = 0, g = 0;
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k;
        if (!(ok = ring_get(ring, t, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        const int nv = kPass == kStatsPass ? 0 : cur.n;
        for (int j = 0; j < nv; ++j, ++g) {
          int n = a.col_idx[cur.first + j];
          n = (n < 0 || n >= a.d.nb) ? 0 : n;
          const int krow = cur.bh * S + n * 128;
          const int vs = g % C::kVStages;
          if (!(ok = mbar_wait(&bars->v_empty[vs], ((g / C::kVStages) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->v_full[vs], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(sV + vs * C::kTile + b * 16384, &tmV, b * 64, krow, &bars->v_full[vs]);
          vg = g + 1;
        }
        if (ok) ring_release(ring, t);
      }
      for (int i = (vg > C::kVStages ? vg - C::kVStages : 0); i < vg; ++i)
        drain_wait(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1);
    }
  } else if (warp == 1 || warp == kWarpPV) {
    // ------------------------------------------------------------ MMAs --
    // Lane 0 of warp 1 issues S = Q K^T of every block as soon as the
    // softmax has taken the previous S out of TMEM; lane 0 of warp 11
    // issues P.V of every block as soon as both halves' P are there.  Each
    // walks the schedule on its own.
    if (lane == 0) {
      const bool s_role = warp == 1;
      const uint32_t idS = instr_desc(Half16<T>::kFmt, 0, 0, 128, 128);
      const uint32_t idPV = instr_desc(Half16<T>::kFmt, 0, 1, D, 128);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      int g = 0, q = 0;  // blocks / non-empty items walked so far
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k = -1;
        if (!(ok = ring_get(ring, t, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        const int qb = q & 1;
        for (int j = 0; j < cur.n && ok; ++j, ++g) {
          if (s_role) {
            const int ks = g % C::kKStages;
            if (j == 0 && !(ok = mbar_wait(&bars->q_full[qb], (q >> 1) & 1, ab, a.status))) break;
            if (!(ok = mbar_wait(&bars->k_full[ks], (g / C::kKStages) & 1, ab, a.status))) break;
            // both warpgroups have loaded S of the previous block
            if (!(ok = mbar_wait(&bars->s_free, (g & 1) ^ 1, ab, a.status))) break;
            tc_fence_after();
            const SDesc dQ(aQ + qb * C::kTile, 16, 1024), dK(aK + ks * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_ss(tmem, dQ.at(off), dK.at(off), idS, kk > 0);
            }
            mma_commit(&bars->k_empty[ks]);
            mma_commit(&bars->s_full);
            if (j == cur.n - 1) mma_commit(&bars->q_empty[qb]);
          } else if constexpr (kPass != kStatsPass) {
            const int vs = g % C::kVStages;
            const int b = g & 1;
            if (!(ok = mbar_wait(&bars->v_full[vs], (g / C::kVStages) & 1, ab, a.status))) break;
            // both halves' P (the first block of a row also overwrites both
            // accumulators, which both warpgroups read while combining the
            // previous row)
            if (!(ok = mbar_wait(&bars->p_full[b], (g >> 1) & 1, ab, a.status))) break;
            tc_fence_after();
            const SDesc dV(aV + vs * C::kTile, 16384, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tmem + kColO + h * D, tmem + kColP + b * 64 + h * 32 + kk * 8,
                            dV.at((4 * h + kk) * 2048), idPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->v_empty[vs]);
            mma_commit(&bars->pv_done[b]);
          }
        }
        if (!ok) break;
        if (cur.n > 0) ++q;
        ring_release(ring, t);
      }
      // every MMA this thread issued has completed before the CTA exits
      uint64_t* fin = &bars->final_mma[s_role ? 0 : 1];
      mma_commit(fin);
      drain_wait(fin, 0);
    }
    __syncwarp();
  } else if (warp < kWarpV) {
    // -------------------------------------------------------- softmax --
    const int hg = (warp - 2) / 4;  // key half of every block
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const uint32_t colO = kColO + hg * D;  // this half's accumulator
    const float sl2 = a.d.scale * kLog2e;
    int g = 0;  // blocks processed by this CTA
    int x = 0;  // row-statistics exchanges (one per non-empty item)
    int sync_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int k = -1;
      if (lane == 0) ok = ring_get(ring, t, &k, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      k = __shfl_sync(0xffffffffu, k, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode_warp(k, cur);
      const int nblk = cur.n;
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      T* orow = (T*)a.O + grow * D + hg * (D / 2);
      if (nblk == 0) {
        if constexpr (kPass != kStatsPass) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D / 16; ++c) ((uint4*)orow)[c] = z;
        }
        if (kPass != kOutPass && hg == 0) {
          a.row_max[grow] = -INFINITY;
          a.row_denom[grow] = 0.f;
        }
        __syncwarp();
        if (lane == 0) ring_release(ring, t);
        continue;
      }
      float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
      if constexpr (kPass == kOutPass) {
        // the row's base-2 log-sum-exp from the statistics pass: P comes
        // out normalised, 2^(scale log2(e) s - lse2)
        m_ref = a.row_max[grow] * kLog2e + log2f(a.row_denom[grow]);
      }
      for (int i = 0; i < nblk; ++i, ++g) {
        const int b = g & 1;
        if (!(ok = warp_wait(&bars->s_full, g & 1, bars, a.status))) break;
        tc_fence_after();
        float tt[64];  // raw scores of this half
        {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + hg * 64, v0);
          tmem_ld32(tmem + lane_base + hg * 64 + 32, v1);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bars->s_free);
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            tt[k] = __uint_as_float(v0[k]);
            tt[32 + k] = __uint_as_float(v1[k]);
          }
        }
        float alpha = 1.f;
        bool rescale = false;
        if constexpr (kPass != kOutPass) {
          // row maximum of this half in log2 units (the scale is applied to
          // the extreme raw score, not to every score)
          const float mx = (sl2 >= 0.f ? extreme64<true>(tt) : extreme64<false>(tt)) * sl2;
          m_true = fmaxf(m_true, mx);
          if (i > 0) {
            const bool need = mx - m_ref > kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
              const float m_new = fmaxf(m_ref, mx);
              alpha = ex2(m_ref - m_new);
              l *= alpha;
              m_ref = m_new;
              rescale = kPass == kOnline;  // the statistics pass keeps no O
            }
          } else {
            m_ref = mx;
          }
        }
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
        uint32_t pk[32];
        const float2 sc = make_float2(sl2, sl2), nm = make_float2(-m_ref, -m_ref);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          // x = s * scale * log2(e) - m_ref in one rounding, then 2^x on MUFU
          const float2 x = fma2(make_float2(tt[2 * k], tt[2 * k + 1]), sc, nm);
          const float2 p = make_float2(ex2(x.x), ex2(x.y));
          sum4[k & 3] = add2(sum4[k & 3], p);
          pk[k] = Half16<T>::pack(p.x, p.y);
        }
        l += (sum4[0].x + sum4[0].y + sum4[1].x + sum4[1].y) + (sum4[2].x + sum4[2].y + sum4[3].x + sum4[3].y);
        if constexpr (kPass == kStatsPass) continue;  // no P, no P.V
        // P of this block goes to buffer b once P.V of block g - 2 (the
        // buffer's previous use) is done; the MMA thread's p_full wait for
        // block g - 2 came before that P.V, so this warpgroup's arrivals on
        // p_full[b] never run two phases ahead of it.  O_h is rescaled only
        // once P.V of block g - 1 is done as well.
        if (g >= 2) {
          if (!(ok = warp_wait(&bars->pv_done[b], ((g >> 1) - 1) & 1, bars, a.status))) break;
          tc_fence_after();
        }
        if (rescale) {
          if (!(ok = warp_wait(&bars->pv_done[b ^ 1], ((g - 1) >> 1) & 1, bars, a.status))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_base + colO + c * 32;
            tmem_ld32(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(ta, v);
          }
        }
        tmem_st32(tmem + lane_base + kColP + b * 64 + hg * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      // ----------------------------------------------------- epilogue --
      // exchange (m_ref, l) of the two halves (and half 1's true max)
      // (the output pass's halves are already normalised: O = O_0 + O_1,
      // which the same combine gives with m = 0, l = 1/2 for both)
      if (x > 0 && !(ok = warp_wait(&bars->red_empty, (x - 1) & 1, bars, a.status))) break;
      sRed[(2 * hg) * 128 + r] = kPass == kOutPass ? 0.f : m_ref;
      sRed[(2 * hg + 1) * 128 + r] = kPass == kOutPass ? 0.5f : l;
      if (hg == 1) sRed[4 * 128 + r] = kPass == kOutPass ? 0.f : m_true;
      mbar_arrive(&bars->red_full);
      if (!(ok = warp_wait(&bars->red_full, x & 1, bars, a.status))) break;
      const float m0 = sRed[r], l0 = sRed[128 + r], m1 = sRed[256 + r], l1 = sRed[384 + r];
      const float mt1 = sRed[512 + r];
      mbar_arrive(&bars->red_empty);
      ++x;
      const float R = fmaxf(m0, m1);
      const float c0 = ex2(m0 - R), c1 = ex2(m1 - R);
      const float L = l0 * c0 + l1 * c1;
      // both halves' last P.V
      if (kPass != kStatsPass && !(ok = warp_wait(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, bars, a.status)))
        break;
      tc_fence_after();
      const uint32_t t0 = tmem + lane_base + kColO + hg * (D / 2);
      if (cur.slot < 0) {
        if constexpr (kPass != kStatsPass) {
          const float inv = 1.f / L;
          const float2 w = make_float2(c0 * inv, c1 * inv);
          // this half's D / 2 output columns as bf16, stored 64 at a time with
          // the rows exchanged in groups of four (st_rows64)
          uint32_t o[D / 4];
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t u[32], v[32];
            tmem_ld32(t0 + c * 32, u);
            tmem_ld32(t0 + D + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 y = fma2(make_float2(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])),
                                    make_float2(w.x, w.x),
                                    mul2(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])),
                                         make_float2(w.y, w.y)));
              o[16 * c + j] = Half16<T>::pack(y.x, y.y);
            }
          }
          if constexpr (D == 128) {
            st_rows64(o, orow, (size_t)D);
          } else {
            st_global_64B(orow, o);
          }
        }
        if (kPass != kOutPass && hg == 0) {
          const float M = fmaxf(m_true, mt1);
          a.row_max[grow] = M * kLn2;
          a.row_denom[grow] = L * ex2(R - M);
        }
      } else {
        // chunk of a split row: publish this half's columns of
        // c0 O_0 + c1 O_1 (relative to R) and the chunk's statistics; the
        // last chunk to arrive combines them:
        //   M = max_c Z_c,  w_c = 2^(R_c - M),  l = sum_c L_c w_c,
        //   O = sum_c w_c O_c / l
        // with Z_c the chunk's true max in half 0 (whose merge writes the row
        // statistics) and R_c in half 1 (any common bound works there).
        constexpr size_t kPart = fwd_part_floats<D>();
        float* tile = a.part + ((size_t)cur.slot * a.d.BH + cur.bh) * kPart;
#pragma unroll 1
        for (int c = 0; c < (kPass == kStatsPass ? 0 : D / 64); ++c) {
          uint32_t u[32], v[32];
          tmem_ld32(t0 + c * 32, u);
          tmem_ld32(t0 + D + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 y = fma2(make_float2(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])), make_float2(c0, c0),
                                  mul2(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])),
                                       make_float2(c1, c1)));
            u[2 * j] = __float_as_uint(y.x);
            u[2 * j + 1] = __float_as_uint(y.y);
          }
          part_store32(tile, hg * (D / 8) + c * 8, r, u);
        }
        const float Z = hg == 0 ? fmaxf(m_true, mt1) : R;
        // the output pass's chunks are already normalised: equal weights
        // 1 / (chunks) make the merge a plain sum
        const float Lc = kPass == kOutPass ? 1.f / (float)lay.line_chunks[lay.slot_line[cur.slot]] : L;
        *(float4*)(tile + 128 * D + (hg * 128 + r) * 4) = make_float4(R, Lc, Z, 0.f);
        bool last = false;
        if (!(ok = merge_arrive(lay, cur.slot, cur.bh, a.d.BH, hg, r, &bars->merge_flag[hg], &bars->wg_sync[hg],
                                sync_phase, ab, a.status, &last)))
          break;
        if (last) {
          const int sl = lay.slot_line[cur.slot];
          const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
          const float* p0 = a.part + ((size_t)base * a.d.BH + cur.bh) * kPart;
          const size_t stride = (size_t)a.d.BH * kPart;  // next chunk, same head
          float M = -INFINITY;
          for (int ch = 0; ch < nc; ++ch) M = fmaxf(M, ld_partial(p0 + ch * stride + 128 * D + (hg * 128 + r) * 4).z);
          float lsum = 0.f;
          for (int ch = 0; ch < nc; ++ch) {
            const float4 st = ld_partial(p0 + ch * stride + 128 * D + (hg * 128 + r) * 4);
            lsum += st.y * ex2(st.x - M);
          }
          const float inv = 1.f / lsum;
#pragma unroll 1
          for (int c = 0; c < (kPass == kStatsPass ? 0 : D / 64); ++c) {
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int ch = 0; ch < nc; ++ch) {
              const float* src = p0 + ch * stride;
              const float w = ex2(ld_partial(src + 128 * D + (hg * 128 + r) * 4).x - M) * inv;
              part_accum32(src, hg * (D / 8) + c * 8, r, w, acc);
            }
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = Half16<T>::pack(acc[2 * j], acc[2 * j + 1]);
            st_global_64B(orow + c * 32, o);
          }
          if (kPass != kOutPass && hg == 0) {
            a.row_max[grow] = M * kLn2;
            a.row_denom[grow] = lsum;
          }
        }
      }
      // this warp's reads of O_0 / O_1 are complete before its warpgroup's
      // next P_h arrival lets the MMA overwrite them
      tc_fence_before();
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

template <typename T, int D, int kPass>
bsr_status launch(const FwdArgs& a, const TensorMaps& tm, cudaStream_t s) {
  using C = Fwd2Cfg<D>;
  auto kern = fwd_tc2_kernel<T, D, kPass>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "fwd_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "fwd_tc: cannot query the SM count");
  LaunchTimer timer(kPass == kOnline ? "fwd_tc" : kPass == kStatsPass ? "fwd2p_stats_tc" : "fwd2p_out_tc", s);
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), C::kSmem, s, tm.q, tm.k, tm.v, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "fwd_tc launch: %s", cudaGetErrorString(e));
  return check_launch("fwd_tc launch");
}

}  // namespace

bool tc_fwd_supported(const Dims& d) {
  return (d.dtype == BSR_BF16 || d.dtype == BSR_F16) && (d.D == 64 || d.D == 128);
}

size_t fwd_part_bytes(int D) {
  return sizeof(float) * (D == 64 ? fwd_part_floats<64>() : fwd_part_floats<128>());
}

template <int kPass>
bsr_status launch_pass(const FwdArgs& a, const TensorMaps& tm, cudaStream_t s) {
  switch (a.d.D) {
    case 64:
      return a.d.dtype == BSR_F16 ? launch<__half, 64, kPass>(a, tm, s) : launch<__nv_bfloat16, 64, kPass>(a, tm, s);
    case 128:
      return a.d.dtype == BSR_F16 ? launch<__half, 128, kPass>(a, tm, s) : launch<__nv_bfloat16, 128, kPass>(a, tm, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "fwd_tc2: head_dim %d", a.d.D);
  }
}

bsr_status launch_fwd_tc2(const FwdArgs& a, cudaStream_t s, int pass) {
  TensorMaps tm;
  bsr_status st = make_tensor_maps(a.d, a.Q, a.K, a.V, &tm);
  if (st != BSR_OK) return st;
  switch (pass) {
    case kOnline: return launch_pass<kOnline>(a, tm, s);
    case kStatsPass: return launch_pass<kStatsPass>(a, tm, s);
    case kOutPass: return launch_pass<kOutPass>(a, tm, s);
    default: return fail(BSR_ERR_INVALID_ARG, "fwd_tc2: pass %d", pass);
  }
}

}  // namespace bsr
