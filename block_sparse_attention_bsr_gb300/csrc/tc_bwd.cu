// Tensor-core backward pass for bf16 operands (head_dim 64 / 128) on sm_103a.
//
// Two kernels, each output tile with exactly one writer and no atomics
// ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.5.1]):
//
//  * dQ (row-first, mirrors the forward, _attn_bwd_dq_kernel): one CTA per
//    block row m of one (batch, head).  For every stored block (m, n):
//        S  = Q_m K_n^T,  dP = dO_m V_n^T                   (tcgen05, TMEM)
//        P  = exp(scale S - row_max) / row_denom,  dS = P * (dP - D_m)
//        dQ_m += dS K_n                                       (tcgen05, TMEM)
//    and dQ_m * scale is stored at the end.
//  * dK/dV (column-first over the BSC lists, _attn_bwd_dkdv_kernel): one CTA
//    per block column n.  For every block row m that stores (m, n):
//        S^T = K_n Q_m^T,  dP^T = V_n dO_m^T
//        P^T, dS^T as above with the statistics of the 128 queries of m
//        dV_n += P^T dO_m,   dK_n += dS^T Q_m
//    and dK_n * scale, dV_n are stored at the end.
//
// The statistics enter as one base-2 log-sum-exp per query,
// lse2 = row_max log2(e) + log2(row_denom), so P = 2^(scale log2(e) S - lse2);
// lse2 and the delta D_i = dO_i . O_i ("trnsparse 0.4.1 -> 0.6.0" diff,
// CHANGELOG [0.5.0]) come from the delta kernel that runs first.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2..9 two elementwise warpgroups.  Thread (warp w, lane l)
// owns TMEM lane 32 (w % 4) + l (a query row in dQ, a key row in dK/dV);
// warpgroup g = (w - 2) / 4 handles columns [64 g, 64 g + 64) of the 128 x 128
// score tiles and half of the output columns in the epilogue.  A warpgroup
// copies its S / dP columns into registers at once and releases them, so the
// MMA of the next block overlaps the elementwise work of this one.  dS (dQ
// kernel) and P^T (dK/dV kernel) go back to TMEM as bf16 and feed the next
// MMA as its A operand from TMEM; dS^T goes to shared memory.
// All waits are bounded (see sm100.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"
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

// Writes 32 consecutive K-elements (bf16) of row r of a 128 x 128 K-major
// operand tile with the 128-byte swizzle: K indices [32 c, 32 c + 32).
__device__ __forceinline__ void st_row_chunk(uint32_t tile, int r, int c, const float* x) {
  const uint32_t row = tile + (c >> 1) * 16384 + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = (c & 1) * 4 + q;  // 16-byte unit inside the 128-byte row
    st_shared_v4(row + ((u ^ (r & 7)) << 4), pack_bf16x2(x[q * 8 + 0], x[q * 8 + 1]),
                 pack_bf16x2(x[q * 8 + 2], x[q * 8 + 3]), pack_bf16x2(x[q * 8 + 4], x[q * 8 + 5]),
                 pack_bf16x2(x[q * 8 + 6], x[q * 8 + 7]));
  }
}

// Stores NC fp32 TMEM columns of this thread's lane (from taddr) as bf16
// times `mul` to global memory at grow.
template <int NC>
__device__ __forceinline__ void store_acc_cols(uint32_t taddr, __nv_bfloat16* grow, float mul) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_wait_ld();
    uint4* dst = (uint4*)(grow + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o;
      o.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * mul, __uint_as_float(v[q * 8 + 1]) * mul);
      o.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * mul, __uint_as_float(v[q * 8 + 3]) * mul);
      o.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * mul, __uint_as_float(v[q * 8 + 5]) * mul);
      o.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * mul, __uint_as_float(v[q * 8 + 7]) * mul);
      dst[q] = o;
    }
  }
}

template <int NC>
__device__ __forceinline__ void zero_cols(__nv_bfloat16* grow) {
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int c = 0; c < NC / 8; ++c) ((uint4*)grow)[c] = z;
}

// Loads 64 fp32 TMEM columns of this lane (two 32-column loads) and waits.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    x[k] = __uint_as_float(a[k]);
    x[32 + k] = __uint_as_float(b[k]);
  }
}

// Packs 64 fp32 values to bf16 pairs and stores them in 32 TMEM columns.
__device__ __forceinline__ void tmem_st_bf16x64(uint32_t taddr, const float (&x)[64]) {
  uint32_t v[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
  tmem_st32(taddr, v);
}

// =================================================================== dQ ====
template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kBarOff = kTile * (2 + 2 * kStages);
  static constexpr int kSmem = kBarOff + 256 + 1024;
};

struct DqBars {
  uint64_t qd_full;
  uint64_t sdp_full;
  uint64_t sdp_free;
  uint64_t ds_full;
  uint64_t dq_done;
  uint64_t final_mma;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  uint32_t tmem_slot;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sdO = sQ + C::kTile;
  uint8_t* sK = sdO + C::kTile;
  uint8_t* sV = sK + C::kStages * C::kTile;
  DqBars* bars = (DqBars*)(sm + C::kBarOff);
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x % a.d.BH;
  const int m = a.row_order[blockIdx.x / a.d.BH];
  const int S = a.d.S;
  const int j0 = a.row_ptr[m];
  const int nblk = a.row_ptr[m + 1] - j0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 1);
    mbar_init(&bars->sdp_full, 1);
    mbar_init(&bars->sdp_free, kEw);
    mbar_init(&bars->ds_full, kEw);
    mbar_init(&bars->dq_done, 1);
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
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

  if (warp == 0) {
    if (lane == 0 && nblk > 0) {
      // ------------------------------------------------------ producer --
      const int qrow = bh * S + m * 128;
      mbar_arrive_expect_tx(&bars->qd_full, 2 * C::kTile);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_2d(sQ + b * 16384, &tmQ, b * 64, qrow, &bars->qd_full);
        tma_load_2d(sdO + b * 16384, &tmdO, b * 64, qrow, &bars->qd_full);
      }
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        int n = a.col_idx[j0 + i];
        if (n < 0 || n >= a.d.nb) {
          atomicExch(a.status, kStatusDeviceCheck);
          n = 0;
        }
        const int krow = bh * S + n * 128;
        const int st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        if (!mbar_wait(&bars->k_empty[st], (use & 1) ^ 1, ab, a.status)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sK + st * C::kTile + b * 16384, &tmK, b * 64, krow, &bars->k_full[st]);
        issued = 2 * i + 1;
        if (!mbar_wait(&bars->v_empty[st], (use & 1) ^ 1, ab, a.status)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sV + st * C::kTile + b * 16384, &tmV, b * 64, krow, &bars->v_full[st]);
        issued = 2 * i + 2;
      }
      drain_wait(&bars->qd_full, 0);
      for (int t = (issued > 2 * C::kStages ? issued - 2 * C::kStages : 0); t < issued; ++t) {
        const int i = t / 2, st = i % C::kStages;
        drain_wait((t & 1) ? &bars->v_full[st] : &bars->k_full[st], (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nblk > 0) {
      // ----------------------------------------------------------- MMA --
      const uint32_t idS = instr_desc(1, 0, 0, 128, 128);
      const uint32_t idDQ = instr_desc(1, 0, 1, D, 128);
      const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(&bars->qd_full, 0, ab, a.status);
      auto issue_sdp = [&](int i) -> bool {
        const int st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        if (!mbar_wait(&bars->k_full[st], use & 1, ab, a.status)) return false;
        if (!mbar_wait(&bars->v_full[st], use & 1, ab, a.status)) return false;
        if (!mbar_wait(&bars->sdp_free, (i & 1) ^ 1, ab, a.status)) return false;
        tc_fence_after();
        const uint32_t kb = aK + st * C::kTile, vb = aV + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColS, smem_desc(aQ + off, 16, 1024), smem_desc(kb + off, 16, 1024), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColDP, smem_desc(adO + off, 16, 1024), smem_desc(vb + off, 16, 1024), idS, kk > 0);
        }
        mma_commit(&bars->v_empty[st]);
        mma_commit(&bars->sdp_full);
        return true;
      };
      if (ok) ok = issue_sdp(0);
      for (int i = 0; ok && i < nblk; ++i) {
        if (i + 1 < nblk && !(ok = issue_sdp(i + 1))) break;
        const int st = i % C::kStages;
        if (!(ok = mbar_wait(&bars->ds_full, i & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t kb = aK + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem + kColDQ, tmem + kColDS + kk * 8, smem_desc(kb + kk * 2048, 16384, 1024), idDQ,
                      (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->k_empty[st]);
        mma_commit(&bars->dq_done);
      }
      mma_commit(&bars->final_mma);
      drain_wait(&bars->final_mma, 0);
    }
  } else {
    // ---------------------------------------------------- elementwise --
    const int g = (warp - 2) / 4;  // column half
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const size_t grow = (size_t)bh * S + (size_t)m * 128 + r;
    __nv_bfloat16* dqrow = (__nv_bfloat16*)a.dQ + grow * D + g * (D / 2);
    if (nblk == 0) {
      zero_cols<D / 2>(dqrow);
    } else {
      const float sl2 = a.d.scale * kLog2e;
      const float lse2 = a.lse2[grow];
      const float dl = a.delta[grow];
      bool ok = true;
      for (int i = 0; i < nblk; ++i) {
        if (!(ok = warp_wait(&bars->sdp_full, i & 1, ab, a.status))) break;
        tc_fence_after();
        float s[64], dp[64];
        tmem_ld64(tmem + lane_base + kColS + g * 64, s);
        tmem_ld64(tmem + lane_base + kColDP + g * 64, dp);
        tc_fence_before();
        mbar_arrive(&bars->sdp_free);
#pragma unroll
        for (int k = 0; k < 64; ++k) s[k] = ex2(fmaf(s[k], sl2, -lse2)) * (dp[k] - dl);
        if (i > 0 && !(ok = warp_wait(&bars->dq_done, (i - 1) & 1, ab, a.status))) break;
        tc_fence_after();
        tmem_st_bf16x64(tmem + lane_base + kColDS + g * 32, s);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->ds_full);
      }
      if (ok) ok = warp_wait(&bars->dq_done, (nblk - 1) & 1, ab, a.status);
      if (ok) {
        tc_fence_after();
        store_acc_cols<D / 2>(tmem + lane_base + kColDQ + g * (D / 2), dqrow, a.d.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================ dK/dV ====
template <int D>
struct DkvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kOp = 128 * 128 * 2;  // dS^T tile
  static constexpr int kBarOff = kTile * (2 + 2 * kStages) + kOp;
  static constexpr int kSmem = kBarOff + 256 + 1024;
};

struct DkvBars {
  uint64_t kv_full;
  uint64_t st_full;
  uint64_t st_free;
  uint64_t pds_full;
  uint64_t pt_free;
  uint64_t dst_free;
  uint64_t final_mma;
  uint64_t q_full[4];
  uint64_t q_empty[4];
  uint64_t do_full[4];
  uint64_t do_empty[4];
  uint32_t tmem_slot;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, BwdArgs a) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = sm;
  uint8_t* sV = sK + C::kTile;
  uint8_t* sQ = sV + C::kTile;
  uint8_t* sdO = sQ + C::kStages * C::kTile;
  uint8_t* sDST = sdO + C::kStages * C::kTile;
  DkvBars* bars = (DkvBars*)(sm + C::kBarOff);
  // P^T (bf16) is written over the dP^T columns each warpgroup has read:
  // queries [0, 64) at column 128, queries [64, 128) at column 192.
  constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 256 + D;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x % a.d.BH;
  const int n = a.col_order[blockIdx.x / a.d.BH];
  const int S = a.d.S;
  const int t0 = a.col_ptr[n];
  const int nblk = a.col_ptr[n + 1] - t0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->st_free, kEw);
    mbar_init(&bars->pds_full, kEw);
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->dst_free, 1);
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->do_full[i], 1);
      mbar_init(&bars->do_empty[i], 1);
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

  if (warp == 0) {
    if (lane == 0 && nblk > 0) {
      // ------------------------------------------------------ producer --
      const int krow = bh * S + n * 128;
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTile);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_2d(sK + b * 16384, &tmK, b * 64, krow, &bars->kv_full);
        tma_load_2d(sV + b * 16384, &tmV, b * 64, krow, &bars->kv_full);
      }
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        int m = a.row_idx[t0 + i];
        if (m < 0 || m >= a.d.nb) {
          atomicExch(a.status, kStatusDeviceCheck);
          m = 0;
        }
        const int qrow = bh * S + m * 128;
        const int st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        if (!mbar_wait(&bars->q_empty[st], (use & 1) ^ 1, ab, a.status)) break;
        mbar_arrive_expect_tx(&bars->q_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sQ + st * C::kTile + b * 16384, &tmQ, b * 64, qrow, &bars->q_full[st]);
        issued = 2 * i + 1;
        if (!mbar_wait(&bars->do_empty[st], (use & 1) ^ 1, ab, a.status)) break;
        mbar_arrive_expect_tx(&bars->do_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sdO + st * C::kTile + b * 16384, &tmdO, b * 64, qrow, &bars->do_full[st]);
        issued = 2 * i + 2;
      }
      drain_wait(&bars->kv_full, 0);
      for (int t = (issued > 2 * C::kStages ? issued - 2 * C::kStages : 0); t < issued; ++t) {
        const int i = t / 2, st = i % C::kStages;
        drain_wait((t & 1) ? &bars->do_full[st] : &bars->q_full[st], (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nblk > 0) {
      // ----------------------------------------------------------- MMA --
      // Per block i: S^T_i and dP^T_i land before the elementwise pass; the
      // elementwise pass reads both and releases them (st_free), so
      // S^T_{i+1} is issued while it computes; P^T_i comes back over the
      // dP^T columns, so dP^T_{i+1} waits for dV_i to finish (pt_free).
      const uint32_t idST = instr_desc(1, 0, 0, 128, 128);
      const uint32_t idG = instr_desc(1, 0, 1, D, 128);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), adO = smem_u32(sdO);
      const uint32_t aDST = smem_u32(sDST);
      auto issue_st = [&](int i) -> bool {
        const int st = i % C::kStages;
        if (!mbar_wait(&bars->q_full[st], (i / C::kStages) & 1, ab, a.status)) return false;
        tc_fence_after();
        const uint32_t qb = aQ + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColST, smem_desc(aK + off, 16, 1024), smem_desc(qb + off, 16, 1024), idST, kk > 0);
        }
        return true;
      };
      auto issue_dpt = [&](int i) -> bool {
        const int st = i % C::kStages;
        if (!mbar_wait(&bars->do_full[st], (i / C::kStages) & 1, ab, a.status)) return false;
        tc_fence_after();
        const uint32_t gb = adO + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColDPT, smem_desc(aV + off, 16, 1024), smem_desc(gb + off, 16, 1024), idST, kk > 0);
        }
        mma_commit(&bars->st_full);
        return true;
      };
      bool ok = mbar_wait(&bars->kv_full, 0, ab, a.status);
      if (ok) ok = issue_st(0) && issue_dpt(0);
      for (int i = 0; ok && i < nblk; ++i) {
        const int st = i % C::kStages;
        if (i + 1 < nblk) {
          if (!(ok = mbar_wait(&bars->st_free, i & 1, ab, a.status))) break;
          if (!(ok = issue_st(i + 1))) break;
        }
        if (!(ok = mbar_wait(&bars->pds_full, i & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t qb = aQ + st * C::kTile, gb = adO + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem + kColDV, tmem + kColDPT + kk * 8 + (kk >= 4 ? 32 : 0),
                      smem_desc(gb + kk * 2048, 16384, 1024), idG, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->pt_free);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColDK, smem_desc(aDST + off, 16, 1024), smem_desc(qb + kk * 2048, 16384, 1024), idG,
                      (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->q_empty[st]);
        mma_commit(&bars->do_empty[st]);
        mma_commit(&bars->dst_free);
        if (i + 1 < nblk) {
          if (!(ok = mbar_wait(&bars->pt_free, i & 1, ab, a.status))) break;
          if (!(ok = issue_dpt(i + 1))) break;
        }
      }
      mma_commit(&bars->final_mma);
      drain_wait(&bars->final_mma, 0);
    }
  } else {
    // ---------------------------------------------------- elementwise --
    const int g = (warp - 2) / 4;  // query half of the tile
    const int wl = warp % 4;
    const int r = wl * 32 + lane;  // key row of the tile
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const size_t grow = (size_t)bh * S + (size_t)n * 128 + r;
    __nv_bfloat16* dkrow = (__nv_bfloat16*)a.dK + grow * D + g * (D / 2);
    __nv_bfloat16* dvrow = (__nv_bfloat16*)a.dV + grow * D + g * (D / 2);
    if (nblk == 0) {
      zero_cols<D / 2>(dkrow);
      zero_cols<D / 2>(dvrow);
    } else {
      const float sl2 = a.d.scale * kLog2e;
      const uint32_t aDST = smem_u32(sDST);
      bool ok = true;
      for (int i = 0; i < nblk; ++i) {
        int m = a.row_idx[t0 + i];
        m = (m < 0 || m >= a.d.nb) ? 0 : m;
        const size_t q0 = (size_t)bh * S + (size_t)m * 128 + g * 64;
        const float4* lse4 = (const float4*)(a.lse2 + q0);
        const float4* dl4 = (const float4*)(a.delta + q0);
        if (!(ok = warp_wait(&bars->st_full, i & 1, ab, a.status))) break;
        tc_fence_after();
        float s[64], dp[64];
        tmem_ld64(tmem + lane_base + kColST + g * 64, s);
        tmem_ld64(tmem + lane_base + kColDPT + g * 64, dp);
        tc_fence_before();
        mbar_arrive(&bars->st_free);
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4) {
          const float4 l = __ldg(lse4 + k4), d = __ldg(dl4 + k4);
          s[4 * k4 + 0] = ex2(fmaf(s[4 * k4 + 0], sl2, -l.x));
          s[4 * k4 + 1] = ex2(fmaf(s[4 * k4 + 1], sl2, -l.y));
          s[4 * k4 + 2] = ex2(fmaf(s[4 * k4 + 2], sl2, -l.z));
          s[4 * k4 + 3] = ex2(fmaf(s[4 * k4 + 3], sl2, -l.w));
          dp[4 * k4 + 0] = s[4 * k4 + 0] * (dp[4 * k4 + 0] - d.x);
          dp[4 * k4 + 1] = s[4 * k4 + 1] * (dp[4 * k4 + 1] - d.y);
          dp[4 * k4 + 2] = s[4 * k4 + 2] * (dp[4 * k4 + 2] - d.z);
          dp[4 * k4 + 3] = s[4 * k4 + 3] * (dp[4 * k4 + 3] - d.w);
        }
        // P^T over this warpgroup's own dP^T columns (already read above;
        // dV of the previous block finished before dP^T of this one began)
        tmem_st_bf16x64(tmem + lane_base + kColDPT + g * 64, s);
        if (i > 0 && !(ok = warp_wait(&bars->dst_free, (i - 1) & 1, ab, a.status))) break;
        st_row_chunk(aDST, r, 2 * g, dp);
        st_row_chunk(aDST, r, 2 * g + 1, dp + 32);
        tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(&bars->pds_full);
      }
      if (ok) ok = warp_wait(&bars->dst_free, (nblk - 1) & 1, ab, a.status);
      if (ok) {
        tc_fence_after();
        store_acc_cols<D / 2>(tmem + lane_base + kColDV + g * (D / 2), dvrow, 1.f);
        store_acc_cols<D / 2>(tmem + lane_base + kColDK + g * (D / 2), dkrow, a.d.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
bsr_status launch_bwd(const BwdArgs& a, const TensorMaps& tm, const CUtensorMap& tmdO, cudaStream_t s) {
  {
    auto kern = dq_tc_kernel<D>;
    const int smem = DqCfg<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "dq_tc: cudaFuncSetAttribute(%d): %s", smem, cudaGetErrorString(e));
    LaunchTimer timer("dq_tc", s);
    kern<<<dim3(a.d.nb * a.d.BH), kThreads, smem, s>>>(tm.q, tm.k, tm.v, tmdO, a);
    bsr_status st = check_launch("dq_tc launch");
    if (st != BSR_OK) return st;
  }
  {
    auto kern = dkdv_tc_kernel<D>;
    const int smem = DkvCfg<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
      return fail(BSR_ERR_CUDA, "dkdv_tc: cudaFuncSetAttribute(%d): %s", smem, cudaGetErrorString(e));
    LaunchTimer timer("dkdv_tc", s);
    kern<<<dim3(a.d.nb * a.d.BH), kThreads, smem, s>>>(tm.q, tm.k, tm.v, tmdO, a);
    return check_launch("dkdv_tc launch");
  }
}

}  // namespace

bool tc_bwd_supported(const Dims& d) { return d.dtype == BSR_BF16 && (d.D == 64 || d.D == 128); }

bsr_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
  if ((((uintptr_t)a.lse2) | ((uintptr_t)a.delta)) & 15)
    return fail(BSR_ERR_INVALID_ARG, "bwd_tc: scratch arrays must be 16-byte aligned");
  TensorMaps tm;
  bsr_status st = make_tensor_maps(a.d, a.Q, a.K, a.V, &tm);
  if (st != BSR_OK) return st;
  CUtensorMap tmdO;
  if ((st = make_tensor_map(a.d, a.dO, &tmdO, "dO")) != BSR_OK) return st;
  switch (a.d.D) {
    case 64: return launch_bwd<64>(a, tm, tmdO, s);
    case 128: return launch_bwd<128>(a, tm, tmdO, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "bwd_tc: head_dim %d", a.d.D);
  }
}

}  // namespace bsr
