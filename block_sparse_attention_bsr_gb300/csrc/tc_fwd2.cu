// Tensor-core forward pass for bf16 operands with head_dim 64 / 128 on
// sm_103a, with P kept in tensor memory.
//
// Same walk as the head_dim-256 kernel in tc_fwd.cu (for each block row m
// of one (batch, head) the row's stored blocks j in [row_ptr[m],
// row_ptr[m+1]) are visited in order and the K / V tiles of block column
// col_idx[j] come straight from HBM by TMA; "trnsparse 0.7.0 -> 0.9.0" diff,
// CHANGELOG [0.8.0], attn_fwd_static), with four changes that keep the
// tensor pipe fed:
//   * persistent CTAs, one per SM, walk the (row, head) work list longest
//     row first (sched.cuh), prefetching the next row's tiles while the
//     current one finishes;
//   * P goes back to tensor memory as bf16 and the P.V MMA reads its A
//     operand from there (no shared-memory round trip for P);
//   * two softmax warpgroups split the 128 columns of each score tile; the
//     row maximum is combined through shared memory;
//   * S is double-buffered in TMEM, so S_{j+1} = Q K_{j+1}^T runs while the
//     softmax of block j is computed.
//
// Warp roles (352 threads): warp 0 TMA producer of Q and K, warp 10 TMA
// producer of V, warp 1 TMEM owner and MMA issuer, warps 2..9 two softmax
// warpgroups; thread (warp w, lane l) owns
// query row 32 (w % 4) + l (its TMEM lane), warpgroup g = (w - 2) / 4 owns
// columns [64 g, 64 g + 64) of the scores and half of O's columns.
// TMEM columns: S buffers at 0 and 128, O at 256 (D columns), P at 384
// (64 columns of bf16 pairs).  All waits are bounded (see sm100.cuh).

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

constexpr int kThreads = 352;  // producer, MMA, 8 softmax warps, V producer
constexpr int kWarpV = 10;
constexpr int kSoftmax = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256, kColP = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max may lag by 2^8

template <int D>
struct Fwd2Cfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kKStages = D == 64 ? 4 : 3;
  static constexpr int kVStages = D == 64 ? 4 : 2;
  static constexpr int kRedOff = kTile * (1 + kKStages + kVStages);
  static constexpr int kBarOff = kRedOff + 2 * 2 * 128 * 4;  // [parity][half][row] maxima
  static constexpr int kSmem = kBarOff + 512 + 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t final_mma;
  uint64_t red_full[2];  // both warpgroups' partial row values written (by parity)
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

// Partial result of one chunk of a split row (fp32): O (128 x D, relative to
// the chunk's reference max) then, per column half and row, the chunk's
// reference max, row sum and true max (log2 units) and a pad.
template <int D>
__host__ __device__ constexpr size_t fwd_part_floats() {
  return (size_t)128 * D + 2 * 128 * 4;
}

// 2^x on the FMA pipe, for x <= 8: x = n + f with n = floor(x), f in [0, 1);
// 2^f ~= 1 + f (c1 + f (c2 + f c3)), a cubic fitted to 2^f on [0, 1] by
// iteratively reweighted least squares on the relative error (max relative
// error 8.6e-5, well below the 2^-9 of the bf16 P it feeds); 2^n is added
// to the exponent bits.  Arguments below -126 are clamped (the result there
// is far below anything a bf16 P can hold next to the row maximum's 1).
__device__ __forceinline__ float exp2_poly(float x) {
  x = fmaxf(x, -126.f);
  const float n = floorf(x);
  const float f = x - n;
  const float p = fmaf(fmaf(fmaf(0.0770655f, f, 0.22764668f), f, 0.6951164f), f, 1.f);
  return __int_as_float(__float_as_int(p) + ((int)n << 23));
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  using C = Fwd2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + C::kTile;
  uint8_t* sV = sK + C::kKStages * C::kTile;
  float* sRed = (float*)(sm + C::kRedOff);
  Bars* bars = (Bars*)(sm + C::kBarOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const PlanLayout lay = plan_layout(a.plan, a.d.nb, (int)gridDim.x, a.d.BH);
  const Walk walk = make_walk(lay, a.d.BH);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], kSoftmax);
    }
    mbar_init(&bars->p_full, kSoftmax);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->red_full[0], kSoftmax);
    mbar_init(&bars->red_full[1], kSoftmax);
    mbar_init(&bars->wg_sync[0], 128);
    mbar_init(&bars->wg_sync[1], 128);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->ring.full[i], 1);
      mbar_init(&bars->ring.empty[i], 2 + kSoftmax / 32);  // MMA, softmax warps, V producer
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
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int k;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &k, ab, a.status)) || k < 0) break;
        Cursor cur;
        walk.decode(k, cur);
        if (cur.n == 0) continue;
        // Q of a new item: the previous item's S MMAs must be done
        if (!(ok = mbar_wait(&bars->q_empty, (q & 1) ^ 1, ab, a.status))) break;
        const int qrow = cur.bh * S + cur.line * 128;
        mbar_arrive_expect_tx(&bars->q_full, C::kTile);
        for (int b = 0; b < C::kBoxes; ++b) tma_load_2d(sQ + b * 16384, &tmQ, b * 64, qrow, &bars->q_full);
        ++q;
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
      if (q > 0) drain_wait(&bars->q_full, (q - 1) & 1);
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
        for (int j = 0; j < cur.n; ++j, ++g) {
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
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA --
      // S of block g+1 (other TMEM buffer) is issued before P.V of block g.
      const uint32_t idS = instr_desc(1, 0, 0, 128, 128);
      const uint32_t idPV = instr_desc(1, 0, 1, D, 128);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      auto issue_s = [&](const Cursor& c) -> bool {
        const int i = c.g;
        const int ks = i % C::kKStages;
        const int b = i & 1;
        if (c.i == 0 && !mbar_wait(&bars->q_full, c.q & 1, ab, a.status)) return false;
        if (!mbar_wait(&bars->k_full[ks], (i / C::kKStages) & 1, ab, a.status)) return false;
        if (!mbar_wait(&bars->s_free[b], ((i >> 1) & 1) ^ 1, ab, a.status)) return false;
        tc_fence_after();
        const uint32_t kb = aK + ks * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + b * 128, smem_desc(aQ + off, 16, 1024), smem_desc(kb + off, 16, 1024), idS, kk > 0);
        }
        mma_commit(&bars->k_empty[ks]);
        mma_commit(&bars->s_full[b]);
        if (c.i == c.n - 1) mma_commit(&bars->q_empty);
        return true;
      };
      bool ok = true;
      auto seek_a = [&](Cursor& c) {
        while (true) {
          int k;
          if (!(ok = ring_get(ring, c.t, &k, ab, a.status)) || k < 0) {
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
          ring_release(ring, c.t);
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
      Cursor A{0, 0, 0, 0, 0, 0, 0, 0, 0, false};
      seek_a(A);
      Cursor B = A;
      if (ok && !A.done) {
        if ((ok = issue_s(A))) next_a(A);
      }
      while (ok && !B.done) {
        if (!A.done) {
          if (!(ok = issue_s(A))) break;
          next_a(A);
          if (!ok) break;
        }
        const int i = B.g;
        const int vs = i % C::kVStages;
        if (!(ok = mbar_wait(&bars->p_full, i & 1, ab, a.status))) break;
        if (!(ok = mbar_wait(&bars->v_full[vs], (i / C::kVStages) & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t vb = aV + vs * C::kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem + kColO, tmem + kColP + kk * 8, smem_desc(vb + kk * 2048, 16384, 1024), idPV,
                      (B.i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->v_empty[vs]);
        mma_commit(&bars->pv_done);
        ++B.g;
        if (++B.i == B.n) {
          ring_release(ring, B.t);
          ++B.q;
          ++B.t;
          seek_b(B);
        }
      }
      mma_commit(&bars->final_mma);
      drain_wait(&bars->final_mma, 0);
    }
  } else if (warp < kWarpV) {
    // -------------------------------------------------------- softmax --
    const int hg = (warp - 2) / 4;  // column half
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const float sl2 = a.d.scale * kLog2e;
    int g = 0;  // blocks processed by this CTA
    int x = 0;  // exchanges through sRed (both warpgroups take part in each)
    int sync_phase = 0;
    bool ok = true;
    // Combines a per-row value of the two column halves through shared
    // memory (two buffers by exchange parity: no thread gets more than one
    // exchange ahead, since each waits for all 256 softmax threads).
    auto exchange = [&](float v, float* other) -> bool {
      float* red = sRed + (x & 1) * 256;
      red[hg * 128 + r] = v;
      mbar_arrive(&bars->red_full[x & 1]);
      const bool good = warp_wait(&bars->red_full[x & 1], (x >> 1) & 1, bars, a.status);
      if (good) *other = red[(hg ^ 1) * 128 + r];
      ++x;
      return good;
    };
    for (int t = 0; ok; ++t) {
      int k = -1;
      if (lane == 0) ok = ring_get(ring, t, &k, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      k = __shfl_sync(0xffffffffu, k, 0);
      if (!ok || k < 0) break;
      Cursor cur;
      walk.decode(k, cur);
      const int nblk = cur.n;
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      __nv_bfloat16* orow = (__nv_bfloat16*)a.O + grow * D + hg * (D / 2);
      if (nblk == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int c = 0; c < D / 16; ++c) ((uint4*)orow)[c] = z;
        if (hg == 0) {
          a.row_max[grow] = -INFINITY;
          a.row_denom[grow] = 0.f;
        }
        __syncwarp();
        if (lane == 0) ring_release(ring, t);
        continue;
      }
      float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
      for (int i = 0; i < nblk; ++i, ++g) {
        const int b = g & 1;
        if (!(ok = warp_wait(&bars->s_full[b], (g >> 1) & 1, bars, a.status))) break;
        tc_fence_after();
        float tt[64];
        {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + b * 128 + hg * 64, v0);
          tmem_ld32(tmem + lane_base + b * 128 + hg * 64 + 32, v1);
          tmem_wait_ld();
          const float2 sc = make_float2(sl2, sl2);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 x0 = mul2(make_float2(__uint_as_float(v0[2 * k]), __uint_as_float(v0[2 * k + 1])), sc);
            const float2 x1 = mul2(make_float2(__uint_as_float(v1[2 * k]), __uint_as_float(v1[2 * k + 1])), sc);
            tt[2 * k] = x0.x;
            tt[2 * k + 1] = x0.y;
            tt[32 + 2 * k] = x1.x;
            tt[32 + 2 * k + 1] = x1.y;
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->s_free[b]);
        // row maximum of this half: eight independent chains, then a tree
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = tt[k];
#pragma unroll
        for (int k = 8; k < 64; ++k) m8[k & 7] = fmaxf(m8[k & 7], tt[k]);
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        float mo;
        if (!(ok = exchange(mx, &mo))) break;
        mx = fmaxf(mx, mo);
        m_true = fmaxf(m_true, mx);
        // The reference max depends only on the scores, so it is settled
        // (and the exponentials computed) before waiting for the previous
        // block's P.V; only the O rescale and the P store have to wait.
        float alpha = 1.f;
        bool rescale = false;
        if (i > 0) {
          const bool need = mx - m_ref > kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(m_ref, mx);
            alpha = ex2(m_ref - m_new);
            l *= alpha;
            m_ref = m_new;
            rescale = true;
          }
        } else {
          m_ref = mx;
        }
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
        uint32_t pk[32];
        const float2 nm = make_float2(-m_ref, -m_ref);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 x = add2(make_float2(tt[2 * k], tt[2 * k + 1]), nm);
          // one pair in four on the FMA pipe, the rest on MUFU (ex2)
          const float2 p = (k & 3) == 3 ? make_float2(exp2_poly(x.x), exp2_poly(x.y)) : make_float2(ex2(x.x), ex2(x.y));
          sum4[k & 3] = add2(sum4[k & 3], p);
          pk[k] = pack_bf16x2(p.x, p.y);
        }
        l += (sum4[0].x + sum4[0].y + sum4[1].x + sum4[1].y) + (sum4[2].x + sum4[2].y + sum4[3].x + sum4[3].y);
        // P.V of the previous block (this row's or the previous row's) must
        // be done before O is rescaled or P is overwritten
        if (g > 0) {
          if (!(ok = warp_wait(&bars->pv_done, (g - 1) & 1, bars, a.status))) break;
          tc_fence_after();
        }
        if (rescale) {
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_base + kColO + hg * (D / 2) + c * 32;
            tmem_ld32(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(ta, v);
          }
        }
        tmem_st32(tmem + lane_base + kColP + hg * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      // ----------------------------------------------------- epilogue --
      // total row sum: the two halves' partial sums share the reference max
      float lo;
      if (!(ok = exchange(l, &lo))) break;
      l += lo;
      if (!(ok = warp_wait(&bars->pv_done, (g - 1) & 1, bars, a.status))) break;
      tc_fence_after();
      if (cur.slot < 0) {
        const float inv = 1.f / l;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kColO + hg * (D / 2) + c * 32, v);
          tmem_wait_ld();
          uint4* dst = (uint4*)(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv);
            o.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv);
            o.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv);
            o.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv);
            dst[q] = o;
          }
        }
        if (hg == 0) {
          a.row_max[grow] = m_true * kLn2;
          a.row_denom[grow] = l * ex2(m_ref - m_true);
        }
      } else {
        // chunk of a split row: publish O (relative to m_ref) and the row's
        // statistics; the last chunk to arrive combines them:
        //   M = max m_true_c,  w_c = 2^(m_ref_c - M),  l = sum l_c w_c,
        //   O = sum w_c O_c / l
        constexpr size_t kPart = fwd_part_floats<D>();
        float* tile = a.part + ((size_t)cur.slot * a.d.BH + cur.bh) * kPart;
        float* prow = tile + (size_t)r * D + hg * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kColO + hg * (D / 2) + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ((float4*)(prow + c * 32))[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
        *(float4*)(tile + 128 * D + (hg * 128 + r) * 4) = make_float4(m_ref, l, m_true, 0.f);
        bool last = false;
        if (!(ok = merge_arrive(lay, cur.slot, cur.bh, a.d.BH, hg, r, &bars->merge_flag[hg], &bars->wg_sync[hg],
                                sync_phase, ab, a.status, &last)))
          break;
        if (last) {
          const int sl = lay.slot_line[cur.slot];
          const int base = lay.line_base[sl], nc = lay.line_chunks[sl];
          const float* t0 = a.part + ((size_t)base * a.d.BH + cur.bh) * kPart;
          const size_t stride = (size_t)a.d.BH * kPart;  // next chunk, same head
          float M = -INFINITY;
          for (int ch = 0; ch < nc; ++ch) M = fmaxf(M, ld_partial(t0 + ch * stride + 128 * D + (hg * 128 + r) * 4).z);
          float lsum = 0.f;
          for (int ch = 0; ch < nc; ++ch) {
            const float4 st = ld_partial(t0 + ch * stride + 128 * D + (hg * 128 + r) * 4);
            lsum += st.y * ex2(st.x - M);
          }
          const float inv = 1.f / lsum;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int ch = 0; ch < nc; ++ch) {
              const float* src = t0 + ch * stride;
              const float w = ex2(ld_partial(src + 128 * D + (hg * 128 + r) * 4).x - M) * inv;
              const float* p = src + (size_t)r * D + hg * (D / 2) + c * 32;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 x4 = ld_partial(p + 4 * j);
                acc[4 * j] = fmaf(w, x4.x, acc[4 * j]);
                acc[4 * j + 1] = fmaf(w, x4.y, acc[4 * j + 1]);
                acc[4 * j + 2] = fmaf(w, x4.z, acc[4 * j + 2]);
                acc[4 * j + 3] = fmaf(w, x4.w, acc[4 * j + 3]);
              }
            }
            uint4* dst = (uint4*)(orow + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16x2(acc[8 * j], acc[8 * j + 1]), pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                                  pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                                  pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
          }
          if (hg == 0) {
            a.row_max[grow] = M * kLn2;
            a.row_denom[grow] = lsum;
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
}

template <int D>
bsr_status launch(const FwdArgs& a, const TensorMaps& tm, cudaStream_t s) {
  using C = Fwd2Cfg<D>;
  auto kern = fwd_tc2_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess)
    return fail(BSR_ERR_CUDA, "fwd_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "fwd_tc: cannot query the SM count");
  LaunchTimer timer("fwd_tc", s);
  kern<<<grid, kThreads, C::kSmem, s>>>(tm.q, tm.k, tm.v, a);
  return check_launch("fwd_tc launch");
}

}  // namespace

size_t fwd_part_bytes(int D) {
  return sizeof(float) * (D == 64 ? fwd_part_floats<64>() : fwd_part_floats<128>());
}

bsr_status launch_fwd_tc2(const FwdArgs& a, cudaStream_t s) {
  TensorMaps tm;
  bsr_status st = make_tensor_maps(a.d, a.Q, a.K, a.V, &tm);
  if (st != BSR_OK) return st;
  switch (a.d.D) {
    case 64: return launch<64>(a, tm, s);
    case 128: return launch<128>(a, tm, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "fwd_tc2: head_dim %d", a.d.D);
  }
}

}  // namespace bsr
