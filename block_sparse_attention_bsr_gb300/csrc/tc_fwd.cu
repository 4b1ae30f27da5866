// Tensor-core forward pass for 16-bit operands (bf16 or fp16; head_dim 256) on
// sm_103a: TMA block walker, tcgen05 MMAs with TMEM accumulators, online
// softmax with the statistics kept on chip.
//
// One CTA owns one block row m of one (batch, head) and walks its stored
// blocks j in [row_ptr[m], row_ptr[m+1]), loading the K and V tiles of block
// column col_idx[j] straight from HBM with TMA (no gather, no padding)
// ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0], attn_fwd_static: one
// launch, statistics on chip, no K/V gather, no host reduction, no per-block
// score round trip through HBM).  head_dim 256 is K-tiled: the Q.K^T
// contraction runs over 64-column chunks of head_dim accumulated into one fp32
// score tile ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.6.0]).  bf16 or
// fp16 operands, fp32 accumulation, fp32 scores and statistics ("trnsparse
// 0.7.0 -> 0.9.0" diff, CHANGELOG [0.9.0]).
//
// Warp roles (256 threads):
//   warp 0      TMA producer (one thread): Q once, then K / V tiles per block
//   warp 1      TMEM owner; one thread issues every tcgen05.mma
//   warps 4..7  softmax: thread r of the warpgroup owns query row r
//               (TMEM lane r), reads S with tcgen05.ld, keeps the running
//               max / sum, writes P (bf16) to shared memory, rescales O in
//               TMEM when the max grows by more than 2^8, and runs the
//               epilogue O / l.
// TMEM columns: S double buffer at 0 and 128, O at 256 (D columns).
//
// Every wait is bounded; a wait that gives up raises the CTA abort flag and
// the device status word (BSR_ERR_TIMEOUT), and the kernel drains its
// in-flight copies and MMAs, frees TMEM and returns.

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

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max allowed to lag by 2^8

template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / 64;                 // 64-column (128-byte) boxes per tile
  static constexpr int kTile = 128 * D * 2;             // bytes of a 128 x D bf16 tile
  static constexpr int kStages = D == 64 ? 4 : (D == 128 ? 2 : 1);
  static constexpr int kP = 128 * 128 * 2;              // P tile (bf16)
  static constexpr int kBarOff = kTile * (1 + 2 * kStages) + kP;
  static constexpr int kSmem = kBarOff + 256 + 1024;    // + barriers + alignment slack
};

struct Bars {
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t final_mma;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Bars* b, int* status) {
  bool ok = mbar_wait(bar, parity, &b->abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + C::kTile;
  uint8_t* sV = sK + C::kStages * C::kTile;
  uint8_t* sP = sV + C::kStages * C::kTile;
  Bars* bars = (Bars*)(sm + C::kBarOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // unsplit plan: work index blockIdx.x is one (block row, head)
  Cursor work;
  make_walk(plan_layout(a.plan, a.d.nb, a.G, a.d.BH), a.d.BH).decode(blockIdx.x, work);
  const int bh = work.bh;
  const int m = work.line;
  const int S = a.d.S;
  const int j0 = a.row_ptr[m];
  const int nblk = a.row_ptr[m + 1] - j0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->pv_done, 1);
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

  if (warp == 0) {
    if (lane == 0 && nblk > 0) {
      // ------------------------------------------------------ producer --
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int qrow = bh * S + m * 128;
      mbar_arrive_expect_tx(&bars->q_full, C::kTile);
      for (int b = 0; b < C::kBoxes; ++b) tma_load_2d(sQ + b * 16384, &tmQ, b * 64, qrow, &bars->q_full);
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
        if (!mbar_wait(&bars->k_empty[st], (use & 1) ^ 1, &bars->abort_flag, a.status)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sK + st * C::kTile + b * 16384, &tmK, b * 64, krow, &bars->k_full[st]);
        if (!mbar_wait(&bars->v_empty[st], (use & 1) ^ 1, &bars->abort_flag, a.status)) {
          issued = i * 2 + 1;
          break;
        }
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_2d(sV + st * C::kTile + b * 16384, &tmV, b * 64, krow, &bars->v_full[st]);
        issued = (i + 1) * 2;
      }
      // drain: every copy issued must have landed before the CTA exits
      mbar_wait(&bars->q_full, 0, &bars->abort_flag, a.status, 200000000ull);
      for (int t = (issued > 2 * C::kStages ? issued - 2 * C::kStages : 0); t < issued; ++t) {
        const int i = t / 2, st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        uint64_t* bar = (t & 1) ? &bars->v_full[st] : &bars->k_full[st];
        // the abort flag may be up already: poll directly with a time bound
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, use & 1) && globaltimer_ns() - t0 < 200000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nblk > 0) {
      // ----------------------------------------------------------- MMA --
      const uint32_t idS = instr_desc(Half16<T>::kFmt, 0, 0, 128, 128);
      const uint32_t idPV = instr_desc(Half16<T>::kFmt, 0, 1, D, 128);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
      bool ok = mbar_wait(&bars->q_full, 0, &bars->abort_flag, a.status);
      auto issue_s = [&](int i) -> bool {
        const int st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        const int b = i & 1;
        if (!mbar_wait(&bars->k_full[st], use & 1, &bars->abort_flag, a.status)) return false;
        if (!mbar_wait(&bars->s_free[b], ((i >> 1) & 1) ^ 1, &bars->abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t kb = aK + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + b * 128, smem_desc(aQ + off, 16, 1024), smem_desc(kb + off, 16, 1024), idS, kk > 0);
        }
        mma_commit(&bars->k_empty[st]);
        mma_commit(&bars->s_full[b]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; ok && i < nblk; ++i) {
        if (i + 1 < nblk && !(ok = issue_s(i + 1))) break;
        const int st = i % C::kStages;
        const uint32_t use = i / C::kStages;
        if (!(ok = mbar_wait(&bars->p_full, i & 1, &bars->abort_flag, a.status))) break;
        if (!(ok = mbar_wait(&bars->v_full[st], use & 1, &bars->abort_flag, a.status))) break;
        tc_fence_after();
        const uint32_t vb = aV + st * C::kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t poff = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + kColO, smem_desc(aP + poff, 16, 1024), smem_desc(vb + kk * 2048, 16384, 1024), idPV,
                      (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->v_empty[st]);
        mma_commit(&bars->pv_done);
      }
      // every MMA issued must complete before TMEM is released
      mma_commit(&bars->final_mma);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->final_mma, 0) && globaltimer_ns() - t0 < 200000000ull) {
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------- softmax --
    const int w = warp - 4;
    const int r = w * 32 + lane;
    const uint32_t lane_base = (uint32_t)(w * 32) << 16;
    const float sl2 = a.d.scale * kLog2e;
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    bool ok = true;
    const uint32_t prow = smem_u32(sP) + r * 128;
    for (int i = 0; i < nblk; ++i) {
      const int b = i & 1;
      if (!(ok = warp_wait(&bars->s_full[b], (i >> 1) & 1, bars, a.status))) break;
      tc_fence_after();
      float t[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + b * 128 + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) t[c * 32 + k] = __uint_as_float(v[k]) * sl2;
      }
      tc_fence_before();
      mbar_arrive(&bars->s_free[b]);
      float mx = t[0];
#pragma unroll
      for (int k = 1; k < 128; ++k) mx = fmaxf(mx, t[k]);
      m_true = fmaxf(m_true, mx);
      if (i > 0) {
        if (!(ok = warp_wait(&bars->pv_done, (i - 1) & 1, bars, a.status))) break;
        tc_fence_after();
        const bool need = mx - m_ref > kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_ref, mx);
          const float alpha = ex2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kColO + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(tmem + lane_base + kColO + c * 32, v);
          }
          tmem_wait_st();
        }
      } else {
        m_ref = mx;
      }
      float sum = 0.f;
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = ex2(t[c16 * 8 + e] - m_ref);
          sum += p[e];
        }
        const uint32_t addr = prow + (c16 >> 3) * 16384 + (((c16 & 7) ^ (r & 7)) << 4);
        st_shared_v4(addr, Half16<T>::pack(p[0], p[1]), Half16<T>::pack(p[2], p[3]), Half16<T>::pack(p[4], p[5]),
                     Half16<T>::pack(p[6], p[7]));
      }
      l += sum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    // ------------------------------------------------------- epilogue --
    const size_t grow = (size_t)bh * S + (size_t)m * 128 + r;
    T* orow = (T*)a.O + grow * D;
    if (ok && nblk > 0) ok = warp_wait(&bars->pv_done, (nblk - 1) & 1, bars, a.status);
    if (ok && nblk > 0) {
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColO + c * 32, v);
        tmem_wait_ld();
        uint4* dst = (uint4*)(orow + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 o;
          o.x = Half16<T>::pack(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv);
          o.y = Half16<T>::pack(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv);
          o.z = Half16<T>::pack(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv);
          o.w = Half16<T>::pack(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv);
          dst[q] = o;
        }
      }
      a.row_max[grow] = m_true * kLn2;
      a.row_denom[grow] = l * ex2(m_ref - m_true);
    } else if (nblk == 0) {
      uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 0; c < D / 8; ++c) ((uint4*)orow)[c] = z;
      a.row_max[grow] = -INFINITY;
      a.row_denom[grow] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int D>
bsr_status launch_fwd(const FwdArgs& a, const TensorMaps& tm, cudaStream_t s) {
  using C = FwdCfg<D>;
  auto kern = fwd_tc_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "fwd_tc: cudaFuncSetAttribute(%d): %s", C::kSmem, cudaGetErrorString(e));
  dim3 grid(a.d.nb * a.d.BH);
  LaunchTimer timer("fwd_tc", s);
  kern<<<grid, kThreads, C::kSmem, s>>>(tm.q, tm.k, tm.v, a);
  return check_launch("fwd_tc launch");
}

}  // namespace

bool tc_fwd_supported(const Dims& d) {
  return (d.dtype == BSR_BF16 || d.dtype == BSR_F16) && (d.D == 64 || d.D == 128 || d.D == 256);
}

bsr_status launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  if (a.d.D <= 128) return launch_fwd_tc2(a, s);
  TensorMaps tm;
  bsr_status st = make_tensor_maps(a.d, a.Q, a.K, a.V, &tm);
  if (st != BSR_OK) return st;
  switch (a.d.D) {
    case 256:
      return a.d.dtype == BSR_F16 ? launch_fwd<__half, 256>(a, tm, s) : launch_fwd<__nv_bfloat16, 256>(a, tm, s);
    default: return fail(BSR_ERR_UNSUPPORTED, "fwd_tc: head_dim %d", a.d.D);
  }
}

}  // namespace bsr
