// Tensor-core kernels for the wide and fp32 cases on sm_103a: bf16 / fp16
// operands with head_dim 256 or 512, and fp32 operands with any head_dim.
//
// One kernel template serves the four walks of the method, each a persistent
// CTA per SM taking (line, head, output slice) work items from the planner's
// queue (sched.cuh):
//
//   mode   walk          per stored block (row tile R = the item's line)        accumulates
//   FWD    block rows    S = Q_m K_n^T,  P = online softmax of scale S          O_m  += P V_n
//   DQ     block rows    S, dP = dO_m V_n^T,  dS = P o (dP - D_m)              dQ_m += dS K_n
//   DV     block cols    S^T = K_n Q_m^T,  P^T = 2^(scale log2e S^T - lse2_m)  dV_n += P^T dO_m
//   DK     block cols    S^T, dP^T = V_n dO_m^T,  dS^T = P^T o (dP^T - D_m)    dK_n += dS^T Q_m
//
// ("trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.8.0]: static walk with the
// statistics on chip and no K/V gather; "trnsparse 0.4.1 -> 0.6.0" diff,
// CHANGELOG [0.5.1]: dQ row-first, dK/dV column-first over the host BSC
// transpose, one writer per output tile; [0.5.0]: the delta identity.)
//
// head_dim is K-tiled: the score contractions (X1 = S or S^T, X2 = dP or
// dP^T) run over 64-column chunks of head_dim accumulated in one fp32 TMEM
// tile ("trnsparse 0.4.1 -> 0.6.0" diff, CHANGELOG [0.6.0]).  The output
// columns are cut into slices of W <= 256 (bf16 / fp16) or W <= 128 (fp32)
// so that the fp32 accumulator fits in TMEM beside the score tiles; each
// slice is a separate work item that recomputes the scores (head_dim 512:
// two slices).  dV and dK run as two launches (their accumulators do not fit
// in one CTA's TMEM together).
//
// fp32 operands run on the same bf16 tensor-core path: each fp32 operand x
// is split into three bf16 pieces x = x0 + x1 + x2 (x0 = bf16(x), x1 =
// bf16(x - x0), x2 = bf16(x - x0 - x1); the residual is below 2^-24 |x|),
// and every product keeps the six piece products a_i b_j with i + j <= 2
// (the "bf16x6" scheme of Henry, Tang and Heinecke, "Leveraging the bfloat16
// artificial intelligence datatype for higher-precision computations",
// ARITH 2019); the dropped terms are below 2^-25 |a b|, the accumulation is
// fp32.  The pieces of Q, K, V, dO are written once per call by split3_kernel;
// P and dS are split the same way by the elementwise warps before they go to
// TMEM.
//
// The tensor cores' fp32 accumulation is not round-to-nearest: every MMA
// into an accumulator of magnitude |s| costs up to about an ulp of |s|, so
// with 6 D / 16 MMAs per score the error grows with head_dim.  The fp32
// kernels therefore keep the scores (S, or S^T in the column walks) in two
// accumulators: the leading products a0 b0 (D / 16 MMAs at full magnitude)
// and the five smaller ones (magnitude 2^-8 |s|), added in registers; the
// forward and the backward compute the scores the same way, so the P the
// backward rebuilds from the forward's statistics stays normalised.  To free
// the TMEM columns this takes, FWD and DV pass P to their accumulate MMAs as
// two pieces, P = p0 + p1 up to 2^-18 |P|, with the five products p_i c_j,
// i + j <= 2.
//
// Operands move in 64-column chunks (128 rows x 128 bytes, 128-byte swizzle,
// 16 KB): the row operand(s) of the item stay resident in shared memory when
// they fit, the other operands of the score contractions stream through a
// ring of chunk slots, and the accumulate operand C (V, K, dO or Q columns of
// the slice) has a buffer of its own loaded by a second producer thread.
//
// Warp roles (352 threads): warp 0 producer of the resident operands and the
// ring, warp 1 TMEM owner and MMA issuer (one elected lane), warps 2..9 two
// elementwise warpgroups (thread (w, l) owns TMEM lane 32 (w % 4) + l, i.e.
// one row of the item's tile; warpgroup h = (w - 2) / 4 takes columns
// [64 h, 64 h + 64) of each score tile and half of the slice's output
// columns), warp 10 producer of C and of the per-block statistics.
// All waits are bounded (sm100.cuh); on expiry the CTA raises its abort flag,
// records BSR_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "kernels.h"
#include "sched.cuh"
#include "sm100.cuh"
#include "tc_common.h"

namespace bsr {
namespace {

using namespace sm100;

constexpr int kFwd = 0, kDq = 1, kDv = 2, kDk = 3;
constexpr int kMapQ = 0, kMapK = 1, kMapV = 2, kMapdO = 3;

constexpr int kWThreads = 352;
constexpr int kWarpC = 10;
constexpr int kEw = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kChunk = 16384;
constexpr int kTileBudget = 224 * 1024;
constexpr int kMaxRing = 12;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: the stale max may lag by 2^8
constexpr int kMinRing = 4;  // ring slots a layout must leave to be preferred

// Which operands stay resident for a whole item: 2 = the row operand R1 (and
// R2 when the mode has a second score contraction), 1 = R1 only, 0 = none;
// the first choice whose leftover ring holds two chunk groups (one group =
// the streamed pieces of one 64-column chunk of a contraction) and at least
// kMinRing slots, else the first that holds one group.
constexpr int wide_residency(int NP, int KC, int WC, bool x2) {
  const int C = NP * WC * kChunk, R = NP * KC * kChunk;
  for (int strict = 1; strict >= 0; --strict) {
    for (int opt = 2; opt >= 0; --opt) {
      if (opt == 1 && !x2) continue;
      const int res = opt == 2 ? R * (x2 ? 2 : 1) : (opt == 1 ? R : 0);
      if (res + C > kTileBudget) continue;
      int ring = (kTileBudget - res - C) / kChunk;
      ring = ring < kMaxRing ? ring : kMaxRing;
      const int g1 = (opt >= 1 ? 0 : NP) + NP;
      const int g2 = x2 ? ((opt == 2 ? 0 : NP) + NP) : 0;
      const int g = g1 > g2 ? g1 : g2;
      if (ring >= (strict ? (2 * g > kMinRing ? 2 * g : kMinRing) : g)) return opt;
    }
  }
  return -1;
}

// Output columns one work item computes: 128 for fp32 operands (three
// pieces each), 256 for 16-bit ones, or head_dim if smaller.
__host__ __device__ constexpr int wide_width(bool f32, int D) {
  return f32 ? (D < 128 ? D : 128) : (D < 256 ? D : 256);
}

// fp32 values of one partial-result tile of a split line: 128 rows x W
// columns, and for the forward the chunk's statistics (reference max, row
// sum, true max, pad) per half and row.
__host__ __device__ constexpr size_t wide_part_floats(int W, bool fwd) {
  return (size_t)128 * W + (fwd ? 2 * 128 * 4 : 0);
}

template <typename T>
struct OpType {
  using type = T;
};
template <>
struct OpType<float> {
  using type = __nv_bfloat16;
};

template <typename T, int D, int MODE>
struct WCfg {
  using Op = typename OpType<T>::type;
  static constexpr int NP = std::is_same<T, float>::value ? 3 : 1;  // operand pieces
  static constexpr bool kX2 = MODE == kDq || MODE == kDk;
  static constexpr bool kZOwn = MODE == kFwd || MODE == kDv;  // Z in its own TMEM columns
  static constexpr int KC = D / 64;
  static constexpr int W = wide_width(NP == 3, D);
  static constexpr int NSL = D / W;
  static constexpr int WC = W / 64;
  static constexpr int kCBytes = NP * WC * kChunk;
  static constexpr int kRBytes = NP * KC * kChunk;
  static constexpr int kRes = wide_residency(NP, KC, WC, kX2);
  static_assert(kRes >= 0, "no shared-memory layout fits");
  static constexpr bool kR1Res = kRes >= 1;
  static constexpr bool kR2Res = kX2 && kRes == 2;
  static constexpr int kResBytes = (kR1Res ? kRBytes : 0) + (kR2Res ? kRBytes : 0);
  static constexpr int kRingRaw = (kTileBudget - kResBytes - kCBytes) / kChunk;
  static constexpr int kRing = kRingRaw < kMaxRing ? kRingRaw : kMaxRing;
  static constexpr int kOffR1 = 0;
  static constexpr int kOffR2 = kOffR1 + (kR1Res ? kRBytes : 0);
  static constexpr int kOffC = kOffR2 + (kR2Res ? kRBytes : 0);
  static constexpr int kOffRing = kOffC + kCBytes;
  static constexpr int kOffAux = kOffRing + kRing * kChunk;  // 2 KB: statistics ring, or the max / sum exchange
  static constexpr int kOffBar = kOffAux + 2048;
  static constexpr int kSmem = kOffBar + 512;
  static_assert(kSmem <= 232448, "shared memory over the per-CTA limit");
  static constexpr int kMapR1 = (MODE == kFwd || MODE == kDq) ? kMapQ : kMapK;
  static constexpr int kMapB1 = (MODE == kFwd || MODE == kDq) ? kMapK : kMapQ;
  static constexpr int kMapR2 = MODE == kDq ? kMapdO : kMapV;
  static constexpr int kMapB2 = MODE == kDq ? kMapV : kMapdO;
  static constexpr int kMapC = MODE == kFwd ? kMapV : (MODE == kDq ? kMapK : (MODE == kDv ? kMapdO : kMapQ));
  // TMEM columns: X1 at 0, X2 (or the Z pieces of FWD / DV) at 128, the
  // accumulator after them
  static constexpr uint32_t kColX1 = 0, kColX2 = 128;
  static constexpr uint32_t kColAcc = (kZOwn && NP == 3) ? 384 : 256;
  static constexpr int kZBufs = (kZOwn && NP == 1) ? 2 : 1;
  // fp32: the X1 scores' smaller piece products in a second accumulator
  // (FWD / DV: columns 256..383, with Z = P in two pieces at 128..255;
  // DQ / DK: columns 384..511, after the accumulator)
  static constexpr bool kSplitS = NP == 3;
  static constexpr uint32_t kColXs = kZOwn ? 256 : 384;
  static constexpr int kZP = (kZOwn && NP == 3) ? 2 : NP;  // pieces of Z
  static_assert(!kSplitS || kColXs + 128 <= kColAcc || kColXs >= kColAcc + W, "score accumulators overlap");
  static_assert(!kSplitS || kColXs + 128 <= kTmemCols, "score accumulator overflows TMEM");
  static_assert(kColAcc + W <= kTmemCols, "accumulator overflows TMEM");
};

// TMEM column of piece p of warpgroup h's half of Z (keys [64 h, 64 h + 64),
// two 16-bit values per column), buffer zb.  FWD / DV keep Z in its own
// columns after X1; DQ / DK write pieces 0 and 1 over the warpgroup's own X1
// columns and piece 2 over its own X2 columns (each already read).
template <int MODE, int NP>
__device__ __forceinline__ uint32_t zcol(int p, int h, int zb) {
  if (MODE == kFwd || MODE == kDv) return NP == 1 ? 128u + 64u * zb + 32u * h : 128u + 64u * p + 32u * h;
  return p < 2 ? 64u * h + 32u * p : 128u + 64u * h;
}

struct WideMaps {
  CUtensorMap m[4][3];  // [Q, K, V, dO][piece]
};

struct WideArgs {
  Dims d;
  const int32_t* idx;  // col_idx (row walks) or row_idx (column walks)
  int32_t* plan;
  void* out;            // O, dQ, dV or dK
  float* row_max;       // FWD
  float* row_denom;     // FWD
  const float* lse2;    // backward: per query row
  const float* delta;   // backward: per query row
  float* part;          // partial results of split lines (wide_part_floats per tile)
  int* status;
  // DK with 16-bit operands on a plan: the dS tiles for the dQ walk over
  // them (dq_ds_kernel, tc_bwd.cu), [BH][nnzb] tiles in BSR order (null: none)
  void* dS;
  const int32_t* bsr_of_bsc;
  int nnzb;
  // DK with 16-bit operands on a plan: the P^T tiles for the dV walk over
  // them (dq_ds_kernel with kDV), [BH][nnzb] tiles in BSC order (null: none)
  void* dP;
};

struct WBars {
  uint64_t r_full, r_empty;
  uint64_t c_full, c_empty;
  uint64_t x1_full, x1_free, x2_full, x2_free;
  uint64_t z_full[2], acc_done[2];
  uint64_t pair_sync;
  uint64_t stat_full[2], stat_empty[2];
  uint64_t final_mma;
  uint64_t ring_full[kMaxRing], ring_empty[kMaxRing];
  uint64_t wg_sync[2];  // each warpgroup's sync around a split line's merge
  RingSmem work;
  int merge_flag[2];
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(WBars) <= 512, "barrier block overflows its shared-memory slot");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 200000000ull) {
  }
}

// Three-way bf16 split of x (x0 + x1 + x2 = x up to 2^-24 |x|).
__device__ __forceinline__ void split3(float x, float& x0, float& x1, float& x2) {
  x0 = __bfloat162float(__float2bfloat16_rn(x));
  const float r = x - x0;
  x1 = __bfloat162float(__float2bfloat16_rn(r));
  x2 = r - x1;
}

// Stores 64 fp32 values of key row r as two bf16 piece tiles, x = x0 + x1
// (x0 = bf16(x), x1 = bf16(x - x0)), at tile and tile + 32 KB (the layout of
// st_tile_sw32_row64), one piece at a time (32 packed words live, not 64).
__device__ __forceinline__ void st_tile_pieces2(uint8_t* tile, int r, int h, const float (&x)[64]) {
  uint32_t v[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
  st_tile_sw32_row64(tile, r, h, v);
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float a0 = __bfloat162float(__float2bfloat16_rn(x[2 * k]));
    const float b0 = __bfloat162float(__float2bfloat16_rn(x[2 * k + 1]));
    v[k] = pack_bf16x2(x[2 * k] - a0, x[2 * k + 1] - b0);
  }
  st_tile_sw32_row64(tile + 128 * 128 * 2, r, h, v);
}

// Writes this warpgroup's 64 values of Z (one per key, fp32) into TMEM as
// ZP pieces of the operand type (pairs of keys per column).
template <typename Op, int MODE, int NP, int ZP>
__device__ __forceinline__ void store_z(uint32_t tbase, int h, int zb, const float (&z)[64]) {
  if constexpr (NP == 1) {
    uint32_t v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = Half16<Op>::pack(z[2 * k], z[2 * k + 1]);
    tmem_st32(tbase + zcol<MODE, NP>(0, h, zb), v);
  } else if constexpr (ZP == 2) {
    uint32_t v0[32], v1[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float a0 = __bfloat162float(__float2bfloat16_rn(z[2 * k]));
      const float b0 = __bfloat162float(__float2bfloat16_rn(z[2 * k + 1]));
      v0[k] = pack_bf16x2(a0, b0);
      v1[k] = pack_bf16x2(z[2 * k] - a0, z[2 * k + 1] - b0);
    }
    tmem_st32(tbase + zcol<MODE, NP>(0, h, zb), v0);
    tmem_st32(tbase + zcol<MODE, NP>(1, h, zb), v1);
  } else {
    uint32_t v0[32], v1[32], v2[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      float a0, a1, a2, b0, b1, b2;
      split3(z[2 * k], a0, a1, a2);
      split3(z[2 * k + 1], b0, b1, b2);
      v0[k] = pack_bf16x2(a0, b0);
      v1[k] = pack_bf16x2(a1, b1);
      v2[k] = pack_bf16x2(a2, b2);
    }
    tmem_st32(tbase + zcol<MODE, NP>(0, h, zb), v0);
    tmem_st32(tbase + zcol<MODE, NP>(1, h, zb), v1);
    tmem_st32(tbase + zcol<MODE, NP>(2, h, zb), v2);
  }
}

// Stores NC accumulator columns (fp32 TMEM, from taddr) of this lane's row
// as T times `mul` at p.
template <int NC, typename T>
__device__ __forceinline__ void store_out(uint32_t taddr, T* p, float mul, size_t ld) {
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll 1
    for (int c = 0; c < NC / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(taddr + c * 32, v);
      tmem_wait_ld();
      float4* dst = (float4*)(p + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(v[4 * q]) * mul, __uint_as_float(v[4 * q + 1]) * mul,
                             __uint_as_float(v[4 * q + 2]) * mul, __uint_as_float(v[4 * q + 3]) * mul);
    }
  } else {
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
      st_rows64(w, p + c * 64, ld);
    }
    if constexpr (NC % 64 != 0) {
      uint32_t v[32];
      tmem_ld32(taddr + NC - 32, v);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j] = Half16<T>::pack(__uint_as_float(v[2 * j]) * mul, __uint_as_float(v[2 * j + 1]) * mul);
      st_global_64B(p + NC - 32, w);
    }
  }
}

template <typename T, int NC>
__device__ __forceinline__ void zero_out(T* p) {
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int c = 0; c < NC * (int)sizeof(T) / 16; ++c) ((uint4*)p)[c] = z;
}

// Sums NC columns of row r (from column group cg0) over the nc partial tiles
// of a split line, chunk ch weighted by wgt(ch), times mul, and stores them
// as T at dst.
template <int NC, typename T, typename Wf>
__device__ __forceinline__ void merge_out(const float* tile0, size_t stride, int nc, int cg0, int r, T* dst, float mul,
                                          Wf wgt) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    for (int ch = 0; ch < nc; ++ch) part_accum32(tile0 + ch * stride, cg0 + c * 8, r, wgt(ch), acc);
    if constexpr (std::is_same<T, float>::value) {
      float4* q = (float4*)(dst + c * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        q[j] = make_float4(acc[4 * j] * mul, acc[4 * j + 1] * mul, acc[4 * j + 2] * mul, acc[4 * j + 3] * mul);
    } else {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = Half16<T>::pack(acc[2 * j] * mul, acc[2 * j + 1] * mul);
      // 128-bit stores: inside the out-of-line split epilogue, the 256-bit
      // form (st_global_64B) was measured to land only the first word of
      // each 32 bytes on the head_dim-256 kernels
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ((uint4*)(dst + c * 32))[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
}

// Epilogue of one chunk of a split line, for warpgroup half hg, row r:
// publishes the half's fp32 partial (the forward's relative to the chunk's
// reference max m_ref, with the chunk's row statistics m_ref, L and m_true);
// the last chunk to arrive (for this head, slice and half) sums them all in
// chunk order into the output:
//   forward:  M = max_c m_true_c, w_c = 2^(m_ref_c - M), l = sum_c L_c w_c,
//             O = sum_c w_c O_c / l, row_max = M ln 2, row_denom = l;
//   backward: the plain sum times mul.
// Cold next to the block loop, so kept out of line: the loop's registers do
// not carry the merge's.  False if a wait gave up.
template <typename T, int MODE, int W>
__device__ __noinline__ bool split_epilogue(const PlanLayout lay, float* part, int slot, int bhp, int BHp, int hg,
                                            int r, uint32_t tacc, T* orow, float mul, float m_ref, float L,
                                            float m_true, float* row_max, float* row_denom, int* merge_flag,
                                            uint64_t* wg_sync, int* merge_phase, volatile int* ab, int* status) {
  constexpr size_t kTileF = wide_part_floats(W, MODE == kFwd);
  float* tile = part + ((size_t)slot * BHp + bhp) * kTileF;
  store_acc_part<W / 2>(tacc, tile, hg * (W / 8), r);
  if constexpr (MODE == kFwd) *(float4*)(tile + 128 * W + (hg * 128 + r) * 4) = make_float4(m_ref, L, m_true, 0.f);
  bool last = false;
  if (!merge_arrive(lay, slot, bhp, BHp, hg, r, merge_flag, wg_sync, *merge_phase, ab, status, &last)) return false;
  if (!last) return true;
  const int sln = lay.slot_line[slot];
  const int nc = lay.line_chunks[sln];
  const float* p0 = part + ((size_t)lay.line_base[sln] * BHp + bhp) * kTileF;
  const size_t stride = (size_t)BHp * kTileF;
  if constexpr (MODE == kFwd) {
    const size_t so = 128 * W + (hg * 128 + r) * 4;
    float M = -INFINITY;
    for (int ch = 0; ch < nc; ++ch) M = fmaxf(M, ld_partial(p0 + ch * stride + so).z);
    float lsum = 0.f;
    for (int ch = 0; ch < nc; ++ch) {
      const float4 st4 = ld_partial(p0 + ch * stride + so);
      lsum += st4.y * ex2(st4.x - M);
    }
    const float inv = 1.f / lsum;
    merge_out<W / 2, T>(p0, stride, nc, hg * (W / 8), r, orow, 1.f,
                        [&](int ch) { return ex2(ld_partial(p0 + ch * stride + so).x - M) * inv; });
    if (row_max) {
      *row_max = M * kLn2;
      *row_denom = lsum;
    }
  } else {
    merge_out<W / 2, T>(p0, stride, nc, hg * (W / 8), r, orow, mul, [](int) { return 1.f; });
  }
  return true;
}

template <typename T, int D, int MODE>
__global__ void __launch_bounds__(kWThreads, 1) wide_kernel(const __grid_constant__ WideMaps tm, WideArgs a) {
  // may run as a programmatic dependent: the prologue touches only shared
  // memory and TMEM; global memory waits for the previous grid
  griddep_launch_dependents();
  using C = WCfg<T, D, MODE>;
  using Op = typename C::Op;
  constexpr int NP = C::NP, KC = C::KC, W = C::W, NSL = C::NSL, WC = C::WC;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the layout assumes a 1024-byte aligned base: refuse otherwise
    griddep_wait();
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  uint8_t* sm = smem_raw;
  float* aux = (float*)(sm + C::kOffAux);
  WBars* bars = (WBars*)(sm + C::kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  // The planner sees each output slice of a head as a head of its own
  // (BHp = heads * NSL, slice fastest), so split lines get a merge counter
  // and partial tiles per slice.
  const int BHp = a.d.BH * NSL;
  const PlanLayout lay = plan_layout(a.plan, a.d.nb, (int)gridDim.x, BHp);
  if (warp == 0) plan_prefetch_l2(a.plan, plan_words(a.d.nb, (int)gridDim.x, BHp));

  if (threadIdx.x == 0) {
    mbar_init(&bars->wg_sync[0], 128);
    mbar_init(&bars->wg_sync[1], 128);
    mbar_init(&bars->r_full, 1);
    mbar_init(&bars->r_empty, 1);
    mbar_init(&bars->c_full, 1);
    mbar_init(&bars->c_empty, 1);
    mbar_init(&bars->x1_full, 1);
    mbar_init(&bars->x1_free, kEw);
    mbar_init(&bars->x2_full, 1);
    mbar_init(&bars->x2_free, kEw);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->z_full[i], kEw);
      mbar_init(&bars->acc_done[i], 1);
      mbar_init(&bars->stat_full[i], 1);
      mbar_init(&bars->stat_empty[i], kEw);
    }
    mbar_init(&bars->pair_sync, kEw);
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&bars->ring_full[i], 1);
      mbar_init(&bars->ring_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->work.full[i], 1);
      mbar_init(&bars->work.empty[i], 2 + kEw / 32);  // MMA warp, C producer, elementwise warps
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
  const Walk walk = make_walk(lay, BHp);
  const int total = walk.total;
  // work index -> item, head and output slice
  auto decode = [&](int w, Cursor& c, int& slice) {
    walk.decode(w, c);
    slice = c.bh % NSL;
    c.bh /= NSL;
  };
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->work;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      int q = 0;          // non-empty items loaded
      uint32_t slot = 0;  // ring chunks issued
      bool ok = true;
      auto load_slot = [&](int map, int piece, int chunk, int row) -> bool {
        const int s = slot % C::kRing;
        if (!mbar_wait(&bars->ring_empty[s], ((slot / C::kRing) & 1) ^ 1, ab, a.status)) return false;
        mbar_arrive_expect_tx(&bars->ring_full[s], kChunk);
        tma_load_2d(sm + C::kOffRing + s * kChunk, &tm.m[map][piece], chunk * 64, row, &bars->ring_full[s]);
        ++slot;
        return true;
      };
      for (int t = 0; ok; ++t) {
        int w;
        if (!(ok = ring_put(ring, t, lay.header + 1, total, &w, ab, a.status)) || w < 0) break;
        Cursor cur;
        int slice;
        decode(w, cur, slice);
        if (cur.n == 0) continue;
        const int lrow = cur.bh * S + cur.line * 128;
        if constexpr (C::kR1Res) {
          // the resident operands of a new item once the previous item's
          // last score MMAs are done with them
          if (!(ok = mbar_wait(&bars->r_empty, (q & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->r_full, C::kResBytes);
          for (int p = 0; p < NP; ++p)
            for (int c = 0; c < KC; ++c)
              tma_load_2d(sm + C::kOffR1 + (p * KC + c) * kChunk, &tm.m[C::kMapR1][p], c * 64, lrow, &bars->r_full);
          if constexpr (C::kR2Res) {
            for (int p = 0; p < NP; ++p)
              for (int c = 0; c < KC; ++c)
                tma_load_2d(sm + C::kOffR2 + (p * KC + c) * kChunk, &tm.m[C::kMapR2][p], c * 64, lrow,
                            &bars->r_full);
          }
        }
        ++q;
        for (int i = 0; i < cur.n && ok; ++i) {
          int pl = a.idx[cur.first + i];
          if (pl < 0 || pl >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            pl = 0;
          }
          const int prow = cur.bh * S + pl * 128;
          // per block: the chunk groups of X2 (if any), then those of X1,
          // in the order the MMA thread consumes them
          if constexpr (C::kX2) {
            for (int c = 0; c < KC && ok; ++c) {
              if constexpr (!C::kR2Res)
                for (int p = 0; p < NP && ok; ++p) ok = load_slot(C::kMapR2, p, c, lrow);
              for (int p = 0; p < NP && ok; ++p) ok = load_slot(C::kMapB2, p, c, prow);
            }
          }
          for (int c = 0; c < KC && ok; ++c) {
            if constexpr (!C::kR1Res)
              for (int p = 0; p < NP && ok; ++p) ok = load_slot(C::kMapR1, p, c, lrow);
            for (int p = 0; p < NP && ok; ++p) ok = load_slot(C::kMapB1, p, c, prow);
          }
        }
      }
      // drain: every copy issued must land before the CTA exits
      if (C::kR1Res && q > 0) drain_wait(&bars->r_full, (q - 1) & 1);
      for (uint32_t i = (slot > (uint32_t)C::kRing ? slot - C::kRing : 0); i < slot; ++i)
        drain_wait(&bars->ring_full[i % C::kRing], (i / C::kRing) & 1);
    }
  } else if (warp == kWarpC) {
    if (lane == 0) {
      // ---------------------------------------------- C / stats producer --
      int g = 0, cg = 0, sg = 0;  // blocks walked, C loads and statistics loads issued
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int w;
        if (!(ok = ring_get(ring, t, &w, ab, a.status)) || w < 0) break;
        Cursor cur;
        int sl;
        decode(w, cur, sl);
        for (int i = 0; i < cur.n; ++i, ++g) {
          int pl = a.idx[cur.first + i];
          pl = (pl < 0 || pl >= a.d.nb) ? 0 : pl;
          const int prow = cur.bh * S + pl * 128;
          // C of block g once the accumulate MMA of block g - 1 is done
          if (!(ok = mbar_wait(&bars->c_empty, (g & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->c_full, C::kCBytes);
          for (int p = 0; p < NP; ++p)
            for (int c = 0; c < WC; ++c)
              tma_load_2d(sm + C::kOffC + (p * WC + c) * kChunk, &tm.m[C::kMapC][p], sl * W + c * 64, prow,
                          &bars->c_full);
          cg = g + 1;
          if constexpr (MODE == kDv || MODE == kDk) {
            // lse2 and delta of the block's 128 queries
            const int ss = g & 1;
            if (!(ok = mbar_wait(&bars->stat_empty[ss], ((g >> 1) & 1) ^ 1, ab, a.status))) break;
            mbar_arrive_expect_tx(&bars->stat_full[ss], 1024);
            bulk_load(aux + ss * 256, a.lse2 + prow, 512, &bars->stat_full[ss]);
            bulk_load(aux + ss * 256 + 128, a.delta + prow, 512, &bars->stat_full[ss]);
            sg = g + 1;
          }
        }
        if (!ok) break;
        ring_release(ring, t);
      }
      if (cg > 0) drain_wait(&bars->c_full, (cg - 1) & 1);
      for (int i = (sg > 2 ? sg - 2 : 0); i < sg; ++i) drain_wait(&bars->stat_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA --
    // The whole warp walks the schedule (descriptor arithmetic stays
    // warp-uniform); one elected lane issues the MMAs and commits.
    const uint32_t leader = elect_one();
    const uint32_t idX = instr_desc(Half16<Op>::kFmt, 0, 0, 128, 128);
    const uint32_t idAcc = instr_desc(Half16<Op>::kFmt, 0, 1, W, 128);
    const uint32_t base = smem_u32(sm);
    uint32_t slot = 0;  // ring chunks consumed, in the producer's order
    bool ok = true;
    auto seek_a = [&](Cursor& c) {
      while (true) {
        int w0 = -1;
        bool good = true;
        if (lane == 0) good = ring_get(ring, c.t, &w0, ab, a.status);
        ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        const int w = __shfl_sync(0xffffffffu, w0, 0);
        if (!ok || w < 0) {
          c.done = true;
          return;
        }
        int slice;
        decode(w, c, slice);
        if (c.n > 0) {
          c.i = 0;
          return;
        }
        ++c.t;
      }
    };
    auto seek_b = [&](Cursor& c) {
      while (true) {
        const int w = *(volatile int32_t*)&ring->k[c.t % kRing];
        if (w < 0) {
          c.done = true;
          return;
        }
        int slice;
        decode(w, c, slice);
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
    // One 64-column chunk of a score contraction into TMEM column colD: the
    // piece products A_i B_j (i + j < NP) over the chunk's 64 columns (with
    // `split` the products other than A_0 B_0 into column kColXs).
    auto x_chunk = [&](uint32_t colD, uint32_t resA, bool streamA, int c, bool first, bool split) -> bool {
      uint32_t aa[NP], bb[NP];
      const uint32_t s0 = slot;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        if (streamA) {
          const int s = slot % C::kRing;
          if (!warp_wait(&bars->ring_full[s], (slot / C::kRing) & 1, ab, a.status)) return false;
          aa[p] = base + C::kOffRing + s * kChunk;
          ++slot;
        } else {
          aa[p] = resA + (p * KC + c) * kChunk;
        }
      }
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const int s = slot % C::kRing;
        if (!warp_wait(&bars->ring_full[s], (slot / C::kRing) & 1, ab, a.status)) return false;
        bb[p] = base + C::kOffRing + s * kChunk;
        ++slot;
      }
      tc_fence_after();
      int term = 0;
#pragma unroll
      for (int i = 0; i < NP; ++i) {
#pragma unroll
        for (int j = 0; j + i < NP; ++j, ++term) {
          const SDesc da(aa[i], 16, 1024), db(bb[j], 16, 1024);
          const bool small = split && term > 0;
          const int first_term = small ? 1 : 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_by(leader, tmem + (small ? C::kColXs : colD), da.at(kk * 32), db.at(kk * 32), idX,
                      (first && term == first_term && kk == 0) ? 0u : 1u);
        }
      }
      for (uint32_t x = s0; x < slot; ++x) mma_commit_by(leader, &bars->ring_empty[x % C::kRing]);
      return true;
    };
    auto issue_x2 = [&](const Cursor& c) -> bool {
      if constexpr (C::kX2) {
        if (c.i == 0 && C::kR1Res && !warp_wait(&bars->r_full, c.q & 1, ab, a.status)) return false;
        if (c.g > 0) {
          // NP == 1: dP of the previous block has been read; NP == 3: its
          // accumulate MMA (which read Z piece 2 over these columns) is done
          if (NP == 1 && !warp_wait(&bars->x2_free, (c.g - 1) & 1, ab, a.status)) return false;
          if (NP == 3 && !warp_wait(&bars->acc_done[(c.g - 1) & 1], ((c.g - 1) >> 1) & 1, ab, a.status))
            return false;
        }
        for (int cc = 0; cc < KC; ++cc)
          if (!x_chunk(C::kColX2, base + C::kOffR2, !C::kR2Res, cc, cc == 0, false)) return false;
        mma_commit_by(leader, &bars->x2_full);
      }
      return true;
    };
    auto issue_x1 = [&](const Cursor& c) -> bool {
      if (!C::kX2 && c.i == 0 && C::kR1Res && !warp_wait(&bars->r_full, c.q & 1, ab, a.status)) return false;
      if (c.g > 0) {
        // FWD / DV: the previous scores are in registers; DQ / DK: the
        // previous accumulate MMA (which read Z over these columns) is done
        if (C::kZOwn && !warp_wait(&bars->x1_free, (c.g - 1) & 1, ab, a.status)) return false;
        if (!C::kZOwn && !warp_wait(&bars->acc_done[(c.g - 1) & 1], ((c.g - 1) >> 1) & 1, ab, a.status))
          return false;
      }
      for (int cc = 0; cc < KC; ++cc)
        if (!x_chunk(C::kColX1, base + C::kOffR1, !C::kR1Res, cc, cc == 0, C::kSplitS)) return false;
      mma_commit_by(leader, &bars->x1_full);
      if (C::kR1Res && c.i == c.n - 1) mma_commit_by(leader, &bars->r_empty);
      return true;
    };
    auto issue_acc = [&](const Cursor& c) -> bool {
      if (!warp_wait(&bars->z_full[c.g & 1], (c.g >> 1) & 1, ab, a.status)) return false;
      if (!warp_wait(&bars->c_full, c.g & 1, ab, a.status)) return false;
      tc_fence_after();
      const int zb = C::kZBufs == 2 ? (c.g & 1) : 0;
      int term = 0;
#pragma unroll
      for (int i = 0; i < C::kZP; ++i) {
#pragma unroll
        for (int j = 0; j + i < NP; ++j, ++term) {
          const SDesc dc(base + C::kOffC + j * WC * kChunk, 16384, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_by(leader, tmem + C::kColAcc, tmem + zcol<MODE, NP>(i, kk >> 2, zb) + (kk & 3) * 8,
                      dc.at(kk * 2048), idAcc, (c.i > 0 || term > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit_by(leader, &bars->c_empty);
      mma_commit_by(leader, &bars->acc_done[c.g & 1]);
      return true;
    };
    Cursor A{0, 0, 0, 0, 0, 0, 0, 0, 0, false};
    seek_a(A);
    Cursor B = A;
    if (ok && !A.done) {
      if ((ok = issue_x2(A) && issue_x1(A))) next_a(A);
    }
    while (ok && !B.done) {
      // When the next block starts another item, this item's last
      // accumulate MMA goes first: the next item's score MMAs wait for its
      // resident operands to load, and the epilogue must not wait behind them.
      const bool a_later = !A.done && A.i == 0;
      if constexpr (C::kZOwn) {
        // the next block's scores run while this block's P is computed
        if (a_later && !(ok = issue_acc(B))) break;
        if (!A.done) {
          if (!(ok = issue_x1(A))) break;
          next_a(A);
          if (!ok) break;
        }
        if (!a_later && !(ok = issue_acc(B))) break;
      } else if constexpr (NP == 1) {
        // dP of the next block while this block's dS is computed
        if (a_later && !(ok = issue_acc(B))) break;
        if (!A.done && !(ok = issue_x2(A))) break;
        if (!a_later && !(ok = issue_acc(B))) break;
        if (!A.done) {
          if (!(ok = issue_x1(A))) break;
          next_a(A);
          if (!ok) break;
        }
      } else {
        if (!(ok = issue_acc(B))) break;
        if (!A.done) {
          if (!(ok = issue_x2(A) && issue_x1(A))) break;
          next_a(A);
          if (!ok) break;
        }
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
  } else {
    // ------------------------------------------------------ elementwise --
    const int hg = (warp - 2) / 4;  // column half of the score tiles
    const int wl = warp % 4;
    const int r = wl * 32 + lane;   // row of the item's tile
    const uint32_t lb = (uint32_t)(wl * 32) << 16;
    const float sl2 = a.d.scale * kLog2e;
    int g = 0, ps = 0, merge_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int w = -1;
      if (lane == 0) ok = ring_get(ring, t, &w, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!ok || w < 0) break;
      Cursor cur;
      int sl;
      decode(w, cur, sl);
      const int bhp = cur.bh * NSL + sl;  // the planner's head of this item
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      T* orow = (T*)a.out + grow * D + sl * W + hg * (W / 2);
      if (cur.n == 0) {
        zero_out<T, W / 2>(orow);
        if (MODE == kFwd && sl == 0 && hg == 0) {
          a.row_max[grow] = -INFINITY;
          a.row_denom[grow] = 0.f;
        }
        __syncwarp();
        if (lane == 0) ring_release(ring, t);
        continue;
      }
      float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;  // FWD
      float lse_r = 0.f, dl_r = 0.f;                          // DQ
      if constexpr (MODE == kDq) {
        lse_r = a.lse2[grow];
        dl_r = a.delta[grow];
      }
      for (int i = 0; i < cur.n; ++i, ++g) {
        int jb = -1;  // DK on a plan: the BSR position of the block, where its dS tile goes
        if constexpr (MODE == kDk) {
          if (a.dS && sl == 0) {
            jb = a.bsr_of_bsc[cur.first + i];
            if (jb < 0 || jb >= a.nnzb) {
              atomicExch(a.status, kStatusDeviceCheck);
              jb = -1;
            }
          }
        }
        if (!(ok = warp_wait(&bars->x1_full, g & 1, ab, a.status))) break;
        if (C::kX2 && !(ok = warp_wait(&bars->x2_full, g & 1, ab, a.status))) break;
        if ((MODE == kDv || MODE == kDk) && !(ok = warp_wait(&bars->stat_full[g & 1], (g >> 1) & 1, ab, a.status)))
          break;
        tc_fence_after();
        float z[64];
        tmem_ld64(tmem + lb + C::kColX1 + hg * 64, z);
        if constexpr (C::kSplitS) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tmem + lb + C::kColXs + hg * 64 + h * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) z[h * 32 + k] += __uint_as_float(v[k]);
          }
        }
        if constexpr (C::kZOwn) {
          tc_fence_before();
          mbar_arrive(&bars->x1_free);
        }
        const float* st = aux + (g & 1) * 256;  // DV / DK: lse2 [0, 128), delta [128, 256) of the block's queries
        if constexpr (MODE == kFwd) {
          // block maximum in log2 units, shared by both halves of the row
          float mx = z[0];
          if (sl2 >= 0.f) {
#pragma unroll
            for (int k = 1; k < 64; ++k) mx = fmaxf(mx, z[k]);
          } else {
#pragma unroll
            for (int k = 1; k < 64; ++k) mx = fminf(mx, z[k]);
          }
          mx *= sl2;
          aux[(g & 1) * 256 + hg * 128 + r] = mx;
          if (!(ok = group_sync(&bars->pair_sync, ps, ab, a.status))) break;
          mx = fmaxf(mx, aux[(g & 1) * 256 + (hg ^ 1) * 128 + r]);
          m_true = fmaxf(m_true, mx);
          bool rescale = false;
          float alpha = 1.f;
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
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            z[k] = ex2(fmaf(z[k], sl2, -m_ref));
            sum += z[k];
          }
          l += sum;
          // the Z buffer's previous accumulate MMA, and before a rescale the
          // last accumulate MMA into O
          if (C::kZBufs == 2 && g >= 2 &&
              !(ok = warp_wait(&bars->acc_done[g & 1], ((g - 2) >> 1) & 1, ab, a.status)))
            break;
          if ((C::kZBufs == 1 || rescale) && g >= 1 &&
              !(ok = warp_wait(&bars->acc_done[(g - 1) & 1], ((g - 1) >> 1) & 1, ab, a.status)))
            break;
          tc_fence_after();
          if (rescale) {
#pragma unroll 1
            for (int c = 0; c < W / 64; ++c) {
              uint32_t v[32];
              const uint32_t ta = tmem + lb + C::kColAcc + hg * (W / 2) + c * 32;
              tmem_ld32(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
              tmem_st32(ta, v);
            }
          }
        } else {
          float dp[64];
          if constexpr (C::kX2) {
            tmem_ld64(tmem + lb + C::kColX2 + hg * 64, dp);
            if constexpr (NP == 1) {
              tc_fence_before();
              mbar_arrive(&bars->x2_free);
            }
          }
          if constexpr (MODE == kDq) {
#pragma unroll
            for (int k = 0; k < 64; ++k) z[k] = ex2(fmaf(z[k], sl2, -lse_r)) * (dp[k] - dl_r);
          } else {
            // P^T from the block's statistics, four at a time (the auxiliary
            // area is 1024-byte aligned)
#pragma unroll
            for (int k4 = 0; k4 < 16; ++k4) {
              const float4 l4 = *(const float4*)(st + hg * 64 + 4 * k4);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) z[4 * k4 + j] = ex2(fmaf(z[4 * k4 + j], sl2, -lv[j]));
            }
            if constexpr (MODE == kDk) {
              if (a.dP && sl == 0) {
                // P^T of the block, by BSC position, for the dV walk over it
                // (fp32: two bf16 pieces, one tile each)
                const int pp = cur.first + i;
                if (pp < a.nnzb) {
                  if constexpr (NP == 1) {
                    uint32_t v[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = Half16<Op>::pack(z[2 * k], z[2 * k + 1]);
                    st_tile_sw32_row64((uint8_t*)a.dP + ((size_t)cur.bh * a.nnzb + pp) * (128 * 128 * 2), r, hg, v);
                  } else {
                    st_tile_pieces2((uint8_t*)a.dP + ((size_t)cur.bh * a.nnzb + pp) * (2 * 128 * 128 * 2), r, hg, z);
                  }
                } else {
                  atomicExch(a.status, kStatusDeviceCheck);
                }
              }
              // dS^T = P^T (dP^T - D)
#pragma unroll
              for (int k4 = 0; k4 < 16; ++k4) {
                const float4 d4 = *(const float4*)(st + 128 + hg * 64 + 4 * k4);
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) z[4 * k4 + j] *= dp[4 * k4 + j] - dv[j];
              }
            }
          }
          if constexpr (MODE == kDv || MODE == kDk) mbar_arrive(&bars->stat_empty[g & 1]);
          if constexpr (MODE == kDv) {
            if (C::kZBufs == 2 && g >= 2 &&
                !(ok = warp_wait(&bars->acc_done[g & 1], ((g - 2) >> 1) & 1, ab, a.status)))
              break;
            if (C::kZBufs == 1 && g >= 1 &&
                !(ok = warp_wait(&bars->acc_done[(g - 1) & 1], ((g - 1) >> 1) & 1, ab, a.status)))
              break;
            tc_fence_after();
          }
        }
        if constexpr (MODE == kDk && NP == 1) {
          // dS^T as operand-type pairs: into TMEM for dK and, on a plan, into
          // the dS tile of (block row m, this column) for the dQ walk (the
          // first slice's walk only)
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = Half16<Op>::pack(z[2 * k], z[2 * k + 1]);
          tmem_st32(tmem + lb + zcol<MODE, NP>(0, hg, 0), v);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->z_full[g & 1]);
          if (jb >= 0) st_tile_sw32_row64((uint8_t*)a.dS + ((size_t)cur.bh * a.nnzb + jb) * (128 * 128 * 2), r, hg, v);
        } else {
          store_z<Op, MODE, NP, C::kZP>(tmem + lb, hg, C::kZBufs == 2 ? (g & 1) : 0, z);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->z_full[g & 1]);
          if constexpr (MODE == kDk && NP == 3) {
            if (jb >= 0)  // fp32 on a plan: dS as two bf16 pieces (2^-16 |dS|) for dq_ds32_kernel
              st_tile_pieces2((uint8_t*)a.dS + ((size_t)cur.bh * a.nnzb + jb) * (2 * 128 * 128 * 2), r, hg, z);
          }
        }
      }
      if (!ok) break;
      // ------------------------------------------------------- epilogue --
      if (!(ok = warp_wait(&bars->acc_done[(g - 1) & 1], ((g - 1) >> 1) & 1, ab, a.status))) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lb + C::kColAcc + hg * (W / 2);
      float L = 0.f;
      if constexpr (MODE == kFwd) {
        // row sum of both halves (same reference max); the exchange buffer
        // is the one the next block's maximum will use, so a second sync
        // keeps the write of that maximum behind this read
        aux[(g & 1) * 256 + hg * 128 + r] = l;
        if (!(ok = group_sync(&bars->pair_sync, ps, ab, a.status))) break;
        L = l + aux[(g & 1) * 256 + (hg ^ 1) * 128 + r];
        if (!(ok = group_sync(&bars->pair_sync, ps, ab, a.status))) break;
      }
      if (cur.slot < 0) {
        if constexpr (MODE == kFwd) {
          store_out<W / 2, T>(tacc, orow, 1.f / L, (size_t)D);
          if (sl == 0 && hg == 0) {
            a.row_max[grow] = m_true * kLn2;
            a.row_denom[grow] = L * ex2(m_ref - m_true);
          }
        } else {
          store_out<W / 2, T>(tacc, orow, (MODE == kDv) ? 1.f : a.d.scale, (size_t)D);
        }
      } else {
        const bool stats = MODE == kFwd && sl == 0 && hg == 0;
        if (!(ok = split_epilogue<T, MODE, W>(lay, a.part, cur.slot, bhp, BHp, hg, r, tacc, orow,
                                               MODE == kFwd ? 1.f : ((MODE == kDv) ? 1.f : a.d.scale), m_ref, L,
                                               m_true, stats ? a.row_max + grow : nullptr,
                                               stats ? a.row_denom + grow : nullptr, &bars->merge_flag[hg],
                                               &bars->wg_sync[hg], &merge_phase, ab, a.status)))
          break;
      }
      // this warp's reads of the accumulator are complete before its next
      // Z arrival lets the MMA overwrite it
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

// ------------------------------------------------ fp32 dQ over stored dS ----
// fp32 operands on a plan: the dK walk stores dS as two bf16 pieces (dS =
// s0 + s1 to 2^-16 |dS|, one tile each in the layout of st_tile_sw32_row64,
// 64 KB per block), and this walk sums dQ_m = scale sum_n dS_mn K_n with the
// five piece products s_i k_j, i + j <= 2, over the three bf16 pieces k_j of
// K (the products with i + j > 2, and s2, are below 2^-24 |dS K|), smallest
// first, into one fp32 TMEM accumulator.  It replaces the recomputing dQ
// mode (six piece products for each of S and dP and for the accumulate)
// and runs on the same plan: items (block row, head, output slice of W =
// min(D, 128) columns).  The block's two dS tiles (64 KB) come through a
// ring of two stages, K's slice as 64-column chunks of three pieces (48 KB)
// through another; MMAs of N = 64 per chunk.  Warp roles as dq_ds_kernel
// (tc_bwd.cu): warp 0 producer, warp 1 MMA issuer, warps 2..9 the epilogue
// with two TMEM accumulators.
constexpr int kDs32Threads = 320;

template <int D>
struct Ds32Cfg {
  static constexpr int W = D < 128 ? D : 128;
  static constexpr int NSL = D / W;
  static constexpr int KCH = W / 64;          // 64-column chunks of K per slice
  static constexpr int kDsBytes = 2 * 32768;  // the two dS piece tiles of one block
  static constexpr int kKBytes = 3 * 16384;   // the three K pieces of one chunk
  static constexpr int kOffK = 2 * kDsBytes;
  static constexpr int kOffBar = kOffK + 2 * kKBytes;
  static constexpr int kSmem = kOffBar + 512;
  static constexpr uint32_t kCols = 2 * W <= 128 ? 128 : 256;  // two accumulators of W columns
};

struct Ds32Bars {
  uint64_t ds_full[2], ds_empty[2];
  uint64_t k_full[2], k_empty[2];
  uint64_t acc_full[2];   // the item's last MMA into accumulator b is done
  uint64_t acc_empty[2];  // the epilogue has read accumulator b
  uint64_t final_mma;
  uint64_t wg_sync[2];
  RingSmem work;
  int merge_flag[2];
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(Ds32Bars) <= 512, "barrier block overflows its shared-memory slot");

// kDV: dV_n = sum_m P^T_nm dO_m the same way over the two bf16 pieces of
// P^T the dK walk stored (BSC order; read as the K-major A operand with
// 32-byte swizzling, M = keys) and dO's three pieces, on the dV plan.
template <int D, bool kDV>
__global__ void __launch_bounds__(kDs32Threads, 1) dq_ds32_kernel(const __grid_constant__ WideMaps tm, WideArgs a) {
  // runs as a programmatic dependent of the dK walk that stored the tiles:
  // the prologue touches only shared memory and TMEM
  griddep_launch_dependents();
  using C = Ds32Cfg<D>;
  constexpr int W = C::W, NSL = C::NSL, KCH = C::KCH;
  static_assert(C::kSmem <= 232448, "shared memory over the per-CTA limit");
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the layout assumes a 1024-byte aligned base: refuse otherwise
    griddep_wait();
    if (threadIdx.x == 0) atomicExch(a.status, kStatusDeviceCheck);
    return;
  }
  uint8_t* sm = smem_raw;
  Ds32Bars* bars = (Ds32Bars*)(sm + C::kOffBar);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = a.d.S;
  const int BHp = a.d.BH * NSL;
  const PlanLayout lay = plan_layout(a.plan, a.d.nb, (int)gridDim.x, BHp);
  if (warp == 0) plan_prefetch_l2(a.plan, plan_words(a.d.nb, (int)gridDim.x, BHp));

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->ds_full[i], 1);
      mbar_init(&bars->ds_empty[i], 1);
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], kEw);
      mbar_init(&bars->wg_sync[i], 128);
    }
    mbar_init(&bars->final_mma, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars->work.full[i], 1);
      mbar_init(&bars->work.empty[i], 1 + kEw / 32);  // MMA warp + epilogue warps
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
  auto decode = [&](int w, Cursor& c, int& slice) {
    walk.decode(w, c);
    slice = c.bh % NSL;
    c.bh /= NSL;
  };
  const uint32_t tmem = bars->tmem_slot;
  volatile int* ab = &bars->abort_flag;
  RingSmem* ring = &bars->work;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      int g = 0, h = 0;  // blocks and K chunks whose copies were issued
      bool ok = true;
      for (int t = 0; ok; ++t) {
        int w;
        if (!(ok = ring_put(ring, t, lay.header + 1, walk.total, &w, ab, a.status)) || w < 0) break;
        Cursor cur;
        int slice;
        decode(w, cur, slice);
        // the line's tile pairs are consecutive (dS: BSR order; P^T: BSC order)
        const uint8_t* ds = (const uint8_t*)(kDV ? a.dP : a.dS) + ((size_t)cur.bh * a.nnzb + cur.first) * C::kDsBytes;
        for (int i = 0; i < cur.n && ok; ++i, ++g) {
          int n = a.idx[cur.first + i];
          if (n < 0 || n >= a.d.nb) {
            atomicExch(a.status, kStatusDeviceCheck);
            n = 0;
          }
          const int st = g & 1;
          if (!(ok = mbar_wait(&bars->ds_empty[st], ((g >> 1) & 1) ^ 1, ab, a.status))) break;
          mbar_arrive_expect_tx(&bars->ds_full[st], C::kDsBytes);
          for (int q = 0; q < 4; ++q)
            bulk_load(sm + st * C::kDsBytes + q * 16384, ds + (size_t)i * C::kDsBytes + q * 16384, 16384,
                      &bars->ds_full[st]);
          for (int c = 0; c < KCH; ++c, ++h) {
            const int ks = h & 1;
            if (!(ok = mbar_wait(&bars->k_empty[ks], ((h >> 1) & 1) ^ 1, ab, a.status))) break;
            mbar_arrive_expect_tx(&bars->k_full[ks], C::kKBytes);
            for (int p = 0; p < 3; ++p)
              tma_load_2d(sm + C::kOffK + ks * C::kKBytes + p * 16384, &tm.m[kDV ? kMapdO : kMapK][p], slice * W + c * 64,
                          cur.bh * S + n * 128, &bars->k_full[ks]);
          }
        }
      }
      // drain: every copy issued must land before the CTA exits
      for (int i = (g > 2 ? g - 2 : 0); i < g; ++i) drain_wait(&bars->ds_full[i & 1], (i >> 1) & 1);
      for (int i = (h > 2 ? h - 2 : 0); i < h; ++i) drain_wait(&bars->k_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA --
    const uint32_t leader = elect_one();
    const uint32_t idK = instr_desc(1, kDV ? 0 : 1, 1, 64, 128);  // bf16 pieces; A MN-major (dS) or K-major (P^T), N = 64
    const uint32_t base = smem_u32(sm);
    // the five piece products s_i k_j, smallest first
    constexpr int kSi[5] = {1, 0, 1, 0, 0};
    constexpr int kKj[5] = {1, 2, 0, 1, 0};
    int g = 0, h = 0, q = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int w0 = -1;
      bool good = true;
      if (lane == 0) good = ring_get(ring, t, &w0, ab, a.status);
      ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
      const int w = __shfl_sync(0xffffffffu, w0, 0);
      if (!ok || w < 0) break;
      Cursor cur;
      int slice;
      decode(w, cur, slice);
      if (cur.n > 0) {
        const int buf = q & 1;
        if (!(ok = warp_wait(&bars->acc_empty[buf], ((q >> 1) & 1) ^ 1, ab, a.status))) break;
        tc_fence_after();
        for (int i = 0; i < cur.n && ok; ++i, ++g) {
          const int st = g & 1;
          if (!(ok = warp_wait(&bars->ds_full[st], (g >> 1) & 1, ab, a.status))) break;
          tc_fence_after();
          for (int c = 0; c < KCH; ++c, ++h) {
            const int ks = h & 1;
            if (!(ok = warp_wait(&bars->k_full[ks], (h >> 1) & 1, ab, a.status))) break;
            tc_fence_after();
#pragma unroll
            for (int pr = 0; pr < 5; ++pr) {
              const uint64_t dA = kDV ? smem_desc(base + st * C::kDsBytes + kSi[pr] * 32768, 16, 256, 6)
                                      : smem_desc(base + st * C::kDsBytes + kSi[pr] * 32768, 4096, 256, 6);
              const SDesc dK(base + C::kOffK + ks * C::kKBytes + kKj[pr] * 16384, 16384, 1024);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss_by(leader, tmem + buf * W + c * 64, dA + (uint64_t)(kk * (kDV ? 256 : 32)), dK.at(kk * 2048), idK,
                          (i > 0 || pr > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_by(leader, &bars->k_empty[ks]);
          }
          if (!ok) break;
          mma_commit_by(leader, &bars->ds_empty[st]);
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
    const int hg = (warp - 2) / 4;  // column half of the slice
    const int wl = warp % 4;
    const int r = wl * 32 + lane;
    const uint32_t lb = (uint32_t)(wl * 32) << 16;
    int q = 0, merge_phase = 0;
    bool ok = true;
    for (int t = 0; ok; ++t) {
      int w = -1;
      if (lane == 0) ok = ring_get(ring, t, &w, ab, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!ok || w < 0) break;
      Cursor cur;
      int slice;
      decode(w, cur, slice);
      const int bhp = cur.bh * NSL + slice;
      const size_t grow = (size_t)cur.bh * S + (size_t)cur.line * 128 + r;
      float* orow = (float*)a.out + grow * D + slice * W + hg * (W / 2);
      if (cur.n == 0) {
        zero_out<float, W / 2>(orow);
      } else {
        const int buf = q & 1;
        if (!(ok = warp_wait(&bars->acc_full[buf], (q >> 1) & 1, ab, a.status))) break;
        tc_fence_after();
        const uint32_t tacc = tmem + lb + buf * W + hg * (W / 2);
        ++q;
        const float mul = kDV ? 1.f : a.d.scale;
        if (cur.slot < 0) {
          store_out<W / 2, float>(tacc, orow, mul, (size_t)D);
        } else if (!(ok = split_epilogue<float, kDq, W>(lay, a.part, cur.slot, bhp, BHp, hg, r, tacc, orow, mul,
                                                        0.f, 0.f, 0.f, nullptr, nullptr, &bars->merge_flag[hg],
                                                        &bars->wg_sync[hg], &merge_phase, ab, a.status))) {
          break;
        }
        tc_fence_before();
        mbar_arrive(&bars->acc_empty[buf]);
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

template <int D, bool kDV = false>
bsr_status launch_ds32(const WideMaps& tm, const WideArgs& a, int grid, cudaStream_t s) {
  using C = Ds32Cfg<D>;
  auto kern = dq_ds32_kernel<D, kDV>;
  const char* name = kDV ? "dv_ps" : "dq_ds";
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: cudaFuncSetAttribute(%d): %s", name, C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer(name, s);
  e = launch_dependent(kern, dim3(grid), dim3(kDs32Threads), C::kSmem, s, tm, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

// fp32 on a plan: dQ over the stored dS pieces, then (with a.dP) dV over the
// stored P^T pieces.
template <int D>
bsr_status launch_ds32_walks(const WideMaps& tm, const WideArgs& q, const WideArgs& v, int grid, cudaStream_t s) {
  bsr_status st = launch_ds32<D>(tm, q, grid, s);
  if (st != BSR_OK || !v.dP) return st;
  return launch_ds32<D, true>(tm, v, grid, s);
}

// fp32 -> three bf16 pieces, x = x0 + x1 + x2 (see the file comment), for
// `count` tensors of n values each: piece p of tensor t at out + (3 t + p) n.
struct SplitArgs {
  const float* src[4];
  __nv_bfloat16* out;
  size_t n;
  int count;
};

__global__ void __launch_bounds__(256) split3_kernel(SplitArgs s) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t n4 = s.n / 4;
  for (int t = 0; t < s.count; ++t) {
    const float4* src = (const float4*)s.src[t];
    __nv_bfloat16* o0 = s.out + (size_t)(3 * t) * s.n;
    __nv_bfloat16* o1 = o0 + s.n;
    __nv_bfloat16* o2 = o1 + s.n;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
      const float4 v = src[i];
      float a0, a1, a2, b0, b1, b2, c0, c1, c2, d0, d1, d2;
      split3(v.x, a0, a1, a2);
      split3(v.y, b0, b1, b2);
      split3(v.z, c0, c1, c2);
      split3(v.w, d0, d1, d2);
      ((uint2*)o0)[i] = make_uint2(pack_bf16x2(a0, b0), pack_bf16x2(c0, d0));
      ((uint2*)o1)[i] = make_uint2(pack_bf16x2(a1, b1), pack_bf16x2(c1, d1));
      ((uint2*)o2)[i] = make_uint2(pack_bf16x2(a2, b2), pack_bf16x2(c2, d2));
    }
  }
}

// Encodes the maps of the operands `which` (Q, K, V, dO order) into tm:
// fp32 operands as their three bf16 pieces in `pieces`, 16-bit operands
// directly.
bsr_status wide_maps(const Dims& d, const void* const* ops, int nops, const void* pieces, WideMaps* tm) {
  const char* names[4] = {"Q", "K", "V", "dO"};
  const size_t n = (size_t)d.BH * d.S * d.D;
  for (int t = 0; t < nops; ++t) {
    if (d.dtype == BSR_F32) {
      Dims dp = d;
      dp.dtype = BSR_BF16;
      for (int p = 0; p < 3; ++p) {
        bsr_status st =
            make_tensor_map(dp, (const __nv_bfloat16*)pieces + (size_t)(3 * t + p) * n, &tm->m[t][p], names[t]);
        if (st != BSR_OK) return st;
      }
    } else {
      bsr_status st = make_tensor_map(d, ops[t], &tm->m[t][0], names[t]);
      if (st != BSR_OK) return st;
    }
  }
  return BSR_OK;
}

bsr_status launch_split(const Dims& d, const void* const* ops, int nops, void* pieces, cudaStream_t s) {
  SplitArgs sa{};
  for (int t = 0; t < nops; ++t) sa.src[t] = (const float*)ops[t];
  sa.out = (__nv_bfloat16*)pieces;
  sa.n = (size_t)d.BH * d.S * d.D;
  sa.count = nops;
  const int sms = sm_count();
  const size_t want = (sa.n / 4 + 255) / 256;
  const unsigned grid = (unsigned)(want < (size_t)(sms > 0 ? 4 * sms : 1) ? want : (size_t)(sms > 0 ? 4 * sms : 1));
  LaunchTimer timer("split3", s);
  const cudaError_t e = launch_dependent(split3_kernel, dim3(grid ? grid : 1), dim3(256), 0, s, sa);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "split3 launch: %s", cudaGetErrorString(e));
  return check_launch("split3 launch");
}

template <typename T, int D, int MODE>
bsr_status launch_mode(const WideMaps& tm, const WideArgs& a, int grid, cudaStream_t s, const char* name) {
  using C = WCfg<T, D, MODE>;
  auto kern = wide_kernel<T, D, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s: cudaFuncSetAttribute(%d): %s", name, C::kSmem, cudaGetErrorString(e));
  LaunchTimer timer(name, s);
  e = launch_dependent(kern, dim3(grid), dim3(kWThreads), C::kSmem, s, tm, a);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

template <int MODE>
bsr_status dispatch_mode(const WideMaps& tm, const WideArgs& a, int grid, cudaStream_t s, const char* name) {
  const Dims& d = a.d;
  if (d.dtype == BSR_F32) {
    switch (d.D) {
      case 64: return launch_mode<float, 64, MODE>(tm, a, grid, s, name);
      case 128: return launch_mode<float, 128, MODE>(tm, a, grid, s, name);
      case 256: return launch_mode<float, 256, MODE>(tm, a, grid, s, name);
      case 512: return launch_mode<float, 512, MODE>(tm, a, grid, s, name);
      default: break;
    }
  } else if (d.dtype == BSR_BF16) {
    if (d.D == 256) return launch_mode<__nv_bfloat16, 256, MODE>(tm, a, grid, s, name);
    if (d.D == 512) return launch_mode<__nv_bfloat16, 512, MODE>(tm, a, grid, s, name);
  } else if (d.dtype == BSR_F16) {
    if (d.D == 256) return launch_mode<__half, 256, MODE>(tm, a, grid, s, name);
    if (d.D == 512) return launch_mode<__half, 512, MODE>(tm, a, grid, s, name);
  }
  return fail(BSR_ERR_UNSUPPORTED, "%s: dtype %d head_dim %d", name, d.dtype, d.D);
}

}  // namespace

bool wide_supported(const Dims& d) {
  if (d.dtype == BSR_F32) return d.D == 64 || d.D == 128 || d.D == 256 || d.D == 512;
  return (d.dtype == BSR_BF16 || d.dtype == BSR_F16) && (d.D == 256 || d.D == 512);
}

int plan_heads(const Dims& d) {
  if (tc_bwd_supported(d) || !wide_supported(d)) return d.BH;
  return d.BH * (d.D / wide_width(d.dtype == BSR_F32, d.D));
}

size_t part_tile_bytes(const Dims& d, bool fwd) {
  if (tc_bwd_supported(d)) return fwd ? fwd_part_bytes(d.D) : sizeof(float) * 128 * (size_t)d.D;
  return sizeof(float) * wide_part_floats(wide_width(d.dtype == BSR_F32, d.D), fwd);
}

size_t wide_piece_bytes(const Dims& d, int tensors) {
  return d.dtype == BSR_F32 ? (size_t)tensors * 3 * (size_t)d.BH * d.S * d.D * sizeof(__nv_bfloat16) : 0;
}

bsr_status launch_fwd_wide(const FwdArgs& a, cudaStream_t s) {
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "fwd_wide: cannot query the SM count");
  const void* ops[3] = {a.Q, a.K, a.V};
  bsr_status st;
  if (a.d.dtype == BSR_F32 && (st = launch_split(a.d, ops, 3, a.pieces, s)) != BSR_OK) return st;
  WideMaps tm{};
  if ((st = wide_maps(a.d, ops, 3, a.pieces, &tm)) != BSR_OK) return st;
  WideArgs w{a.d, a.col_idx, a.plan, a.O, a.row_max, a.row_denom, nullptr, nullptr, a.part, a.status};
  return dispatch_mode<kFwd>(tm, w, grid, s, "fwd_wide");
}

bsr_status launch_bwd_wide(const BwdArgs& a, cudaStream_t s) {
  const int grid = tc_grid(a.d);
  if (grid <= 0) return fail(BSR_ERR_CUDA, "bwd_wide: cannot query the SM count");
  const void* ops[4] = {a.Q, a.K, a.V, a.dO};
  bsr_status st;
  if (a.d.dtype == BSR_F32 && (st = launch_split(a.d, ops, 4, a.pieces, s)) != BSR_OK) return st;
  WideMaps tm{};
  if ((st = wide_maps(a.d, ops, 4, a.pieces, &tm)) != BSR_OK) return st;
  // partial tiles (split plans only): dQ's at part_q, dV's at part_kv and
  // dK's after them
  const size_t set = a.part_kv ? plan_tiles(a.d.nb, grid, plan_heads(a.d)) * (part_tile_bytes(a.d, false) / 4) : 0;
  const WideArgs q{a.d, a.col_idx, a.row_plan, a.dQ, nullptr, nullptr, a.lse2, a.delta, a.part_q, a.status};
  const WideArgs v{a.d, a.row_idx, a.col_plan, a.dV, nullptr, nullptr, a.lse2, a.delta, a.part_kv, a.status};
  WideArgs k{a.d, a.row_idx, a.col_plan2, a.dK, nullptr, nullptr, a.lse2, a.delta,
             a.part_kv ? a.part_kv + set : nullptr, a.status};
  // dQ, dV and dK read the same inputs and write different outputs; each is
  // a persistent grid of its own work list.  On a plan with 16-bit operands
  // (a.dS) the dK walk stores its dS tiles and the dQ walk runs after it,
  // summing dS K over them (dq_ds_kernel) instead of recomputing the scores.
  if (a.dS) {
    k.dS = a.dS;
    k.bsr_of_bsc = a.bsr_of_bsc;
    k.nnzb = a.nnzb;
    if (a.dP && a.d.dtype != BSR_F32) {
      // 16-bit: the dK walk also stores P^T; dQ and dV then stream dS and P^T
      k.dP = a.dP;
      if ((st = dispatch_mode<kDk>(tm, k, grid, s, "dk_wide")) != BSR_OK) return st;
      if ((st = launch_dq_ds(a, s)) != BSR_OK) return st;
      return launch_dv_ps(a, s);
    }
    if (a.d.dtype != BSR_F32 || !a.dP) {
      if ((st = dispatch_mode<kDv>(tm, v, grid, s, "dv_wide")) != BSR_OK) return st;
    } else {
      k.dP = a.dP;  // fp32: the dK walk also stores P^T (two pieces) for the dV walk below
    }
    if ((st = dispatch_mode<kDk>(tm, k, grid, s, "dk_wide")) != BSR_OK) return st;
    if (a.d.dtype != BSR_F32) return launch_dq_ds(a, s);
    WideArgs q32 = q;  // fp32: the five-product walks over the stored pieces, on the same plans
    q32.dS = a.dS;
    q32.nnzb = a.nnzb;
    WideArgs v32 = v;
    v32.dP = a.dP;
    v32.nnzb = a.nnzb;
    switch (a.d.D) {
      case 64: return launch_ds32_walks<64>(tm, q32, v32, grid, s);
      case 128: return launch_ds32_walks<128>(tm, q32, v32, grid, s);
      case 256: return launch_ds32_walks<256>(tm, q32, v32, grid, s);
      case 512: return launch_ds32_walks<512>(tm, q32, v32, grid, s);
      default: return fail(BSR_ERR_UNSUPPORTED, "dq_ds: fp32 head_dim %d", a.d.D);
    }
  }
  if ((st = dispatch_mode<kDq>(tm, q, grid, s, "dq_wide")) != BSR_OK) return st;
  if ((st = dispatch_mode<kDv>(tm, v, grid, s, "dv_wide")) != BSR_OK) return st;
  return dispatch_mode<kDk>(tm, k, grid, s, "dk_wide");
}

}  // namespace bsr
