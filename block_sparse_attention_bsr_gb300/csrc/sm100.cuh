// Inline-PTX building blocks for the Blackwell (sm_100a / sm_103a) kernels:
// mbarriers with bounded waits, TMA tile loads, TMEM allocation, tcgen05 MMA
// issue / commit, and TMEM <-> register moves.  Everything here is written
// from the PTX ISA's descriptions of these instructions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace bsr {
namespace sm100 {

// ------------------------------------------------------------ addresses --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase of `bar` with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The device status block every kernel receives as `status`: word 0 is the
// status word (kStatusTimeout / kStatusDeviceCheck, read and cleared by the
// host), words 2..3 the limit of the bounded waits in nanoseconds (64-bit,
// default 2 s; the host lowers it only to test the give-up path).
__device__ __forceinline__ uint64_t wait_limit_ns(const int* status) {
  return *(const volatile unsigned long long*)(status + 2);
}

// Waits until the phase of `bar` with the given parity has completed.  Gives
// up after `timeout_ns` of wall time (0: the status block's limit); on
// give-up it records kStatusTimeout in *status, raises the CTA's abort flag
// and returns false.  Once the abort flag is up every later wait returns
// false immediately.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t timeout_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = timeout_ns ? timeout_ns : wait_limit_ns(status);
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicExch(status, 4 /* BSR_ERR_TIMEOUT */);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA --
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled store of one box from shared memory (same box and swizzle as the
// loads) at element coordinates (x, y); completion tracked by bulk groups.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t x, int32_t y, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the shared-memory sources of all committed bulk stores have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until all committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Makes generic-proxy shared-memory writes visible to the async proxy
// (tensor core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------- programmatic dependent launch --
// A kernel launched as a programmatic dependent of the previous kernel in its
// stream may start before that kernel has finished; griddep_wait() blocks
// until the previous grid has completed and its memory operations are
// visible (a no-op for a kernel launched the ordinary way).
// griddep_launch_dependents() lets the next kernel, if launched as a
// programmatic dependent, start launching once every CTA of this grid has
// executed it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- TMEM --
// Allocates `ncols` (power of two, 32..512) TMEM columns; the whole warp must
// call it.  The base address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// -------------------------------------------------------- descriptors --
// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), the fixed version field (1 at bit 46)
// and the swizzle mode in bits 61..63 (0 = none, 2 = 128-byte, 6 = 32-byte
// swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle = 2) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

// The same descriptor split into words for one operand tile: the low word
// holds the start address (>> 4) and LBO, the high word SBO, the fixed
// version bit and the swizzle mode.  A byte offset inside the tile adds
// off >> 4 to the low word (the operand address stays below 256 KB, so the
// 14-bit address field never carries), which keeps the per-MMA descriptor
// arithmetic at one integer add.
struct SDesc {
  uint32_t lo, hi;
  __device__ __forceinline__ SDesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
      : lo(((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16)),
        hi(((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29)) {}
  __device__ __forceinline__ uint64_t at(uint32_t off) const { return ((uint64_t)hi << 32) | (lo + (off >> 4)); }
};

// Instruction descriptor for kind::f16: fp32 accumulator, operand format
// code `ab_fmt` (1 = bf16, 0 = f16), A / B major-ness (0 = K-major,
// 1 = MN-major), N and M.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_fmt, uint32_t a_mn_major, uint32_t b_mn_major,
                                                  uint32_t N, uint32_t M) {
  return (1u << 4)                 // D format: f32
         | (ab_fmt << 7)           // A format
         | (ab_fmt << 10)          // B format
         | (a_mn_major << 15)      // A major
         | (b_mn_major << 16)      // B major
         | ((N >> 3) << 17)        // N / 8
         | ((M >> 4) << 24);       // M / 16
}

// ------------------------------------------------------------------ MMA --
// D[tmem] (+)= A[smem] * B[smem]^T per the descriptors; `accumulate` = 0
// overwrites D.  Issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with the A operand read from TMEM (M = 128 lanes; for 16-bit types
// two consecutive K elements per 32-bit column, the lower one in the low half).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-converged forms: the whole warp executes the call (so descriptor
// arithmetic stays warp-uniform) and only the lane with `leader` != 0 issues
// the operation.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred;
}

__device__ __forceinline__ void mma_ss_by(uint32_t leader, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, l;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 l, %5, 0;\n\t"
      "@l tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}

__device__ __forceinline__ void mma_ts_by(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, l;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 l, %5, 0;\n\t"
      "@l tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}

__device__ __forceinline__ void mma_commit_by(uint32_t leader, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred l;\n\t"
      "setp.ne.b32 l, %1, 0;\n\t"
      "@l tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
      "r"(leader)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// -------------------------------------------------------- TMEM <-> regs --
// 32 lanes x 32 columns of 32-bit values: thread t of the warp gets lane
// (lane base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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

// ------------------------------------------------------------- helpers --
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The 16-bit operand types of the tensor-core kernels: the A / B format
// code of a kind::f16 MMA (A and B always of the same type) and
// round-to-nearest-even packing of two fp32 values, the first in the low
// half.
template <typename T>
struct Half16;
template <>
struct Half16<__nv_bfloat16> {
  static constexpr uint32_t kFmt = 1;
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
};
template <>
struct Half16<__half> {
  static constexpr uint32_t kFmt = 0;
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16x2(lo, hi); }
};

// 256-bit global store (p 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, uint4 lo, uint4 hi) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(lo.x), "r"(lo.y), "r"(lo.z),
               "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
               : "memory");
}

// Stores one key row's 64 16-bit values (w: 32 packed pairs, queries
// [64 h, 64 h + 64) of key r) into a 128 x 128 tile laid out as the MN-major
// MMA operand with 32-byte swizzling (M = queries, K = keys): 32-byte units
// of 16 queries, unit c / 16 of key r at (c / 16) * 4096 + (r / 8) * 256 +
// (r % 8) * 32 bytes from the (1024-byte aligned) tile, its 16-byte halves
// swapped for r % 8 >= 4.  Four 256-bit stores; the 32 lanes of a warp (32
// consecutive keys) fill 1 KB of contiguous memory with each.
__device__ __forceinline__ void st_tile_sw32_row64(uint8_t* tile, int r, int h, const uint32_t (&w)[32]) {
  uint8_t* dst = tile + h * 4 * 4096 + (r / 8) * 256 + (r % 8) * 32;
  const bool swap = (r & 4) != 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 q0 = make_uint4(w[8 * u], w[8 * u + 1], w[8 * u + 2], w[8 * u + 3]);
    const uint4 q1 = make_uint4(w[8 * u + 4], w[8 * u + 5], w[8 * u + 6], w[8 * u + 7]);
    st_global_v8(dst + u * 4096, swap ? q1 : q0, swap ? q0 : q1);
  }
}

// Stores 16 words (32 16-bit values) at p (16-byte aligned): two 256-bit stores when
// p is 32-byte aligned (each then fills whole 32-byte sectors), else four
// 128-bit stores.
__device__ __forceinline__ void st_global_64B(void* p, const uint32_t (&w)[16]) {
  if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"((char*)p + 32 * h),
                   "r"(w[8 * h]), "r"(w[8 * h + 1]), "r"(w[8 * h + 2]), "r"(w[8 * h + 3]), "r"(w[8 * h + 4]),
                   "r"(w[8 * h + 5]), "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                   : "memory");
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) ((uint4*)p)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// Stores 64 16-bit values (32 packed words w) of each of the warp's 32 consecutive
// rows: lane l holds row l, which starts at `row` (its own pointer), rows
// `ld` elements apart.  The four lanes of each group of four rows exchange
// 32-byte chunks (a 4 x 4 block transpose in two shuffle steps: partner
// lanes l ^ 2, then l ^ 1), so each 256-bit store writes 8 rows x 128
// contiguous bytes instead of 32 rows x 32 bytes (a quarter of the
// cache-line touches).  The whole warp calls it; `row` must be 32-byte
// aligned and ld * 2 a multiple of 32 (otherwise rows are stored as they
// are).  w is clobbered.
template <typename T>
__device__ __forceinline__ void st_rows64(uint32_t (&w)[32], T* row, size_t ld) {
  static_assert(sizeof(T) == 2, "16-bit elements");
  const int q = threadIdx.x & 3;
  const bool aligned = ((reinterpret_cast<uintptr_t>(row) & 31) == 0) && ((ld * 2) % 32 == 0);
  if (!__all_sync(0xffffffffu, aligned)) {
    uint32_t h[16];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int j = 0; j < 16; ++j) h[j] = w[16 * c + j];
      st_global_64B(row + 32 * c, h);
    }
    return;
  }
  const bool b1 = (q & 2) != 0, b0 = (q & 1) != 0;
  // chunk c of lane q = words 8 c .. 8 c + 7 = row q, columns 16 c .. 16 c + 15
#pragma unroll
  for (int c = 0; c < 2; ++c) {  // chunks c and c + 2 with lane q ^ 2
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t lo = w[8 * c + j], hi = w[8 * (c + 2) + j];
      const uint32_t r = __shfl_xor_sync(0xffffffffu, b1 ? lo : hi, 2);
      w[8 * c + j] = b1 ? r : lo;
      w[8 * (c + 2) + j] = b1 ? hi : r;
    }
  }
#pragma unroll
  for (int c = 0; c < 4; c += 2) {  // chunks c and c + 1 with lane q ^ 1
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t lo = w[8 * c + j], hi = w[8 * (c + 1) + j];
      const uint32_t r = __shfl_xor_sync(0xffffffffu, b0 ? lo : hi, 1);
      w[8 * c + j] = b0 ? r : lo;
      w[8 * (c + 1) + j] = b0 ? hi : r;
    }
  }
  // lane q now holds, in words 8 k .. 8 k + 7, chunk q of row (l - q) + k
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    T* p = row + (ptrdiff_t)(k - q) * (ptrdiff_t)ld + 16 * q;
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[8 * k]),
                 "r"(w[8 * k + 1]), "r"(w[8 * k + 2]), "r"(w[8 * k + 3]), "r"(w[8 * k + 4]), "r"(w[8 * k + 5]),
                 "r"(w[8 * k + 6]), "r"(w[8 * k + 7])
                 : "memory");
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (two lanes of work per instruction).
// Three-input maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace sm100
}  // namespace bsr
