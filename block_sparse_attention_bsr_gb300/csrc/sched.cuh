// Persistent work distribution shared by the tensor-core kernels.
//
// The grid holds one CTA per SM.  The planner (plan.cu) lists the work items
// of one kernel -- a block row (forward, dQ) or block column (dK/dV), or a
// chunk of one when the line is long -- sorted longest first, and every item
// is done once per (batch, head): a work index k stands for one (item, head)
// pair through the plan's bucket table (Walk::decode).  CTA b takes work
// index b first, then further indices from a global counter that starts at
// the grid size, so an SM that drew a long item takes fewer short ones after
// it (longest-processing-time-first list scheduling; the pages balance their
// two cores "by stored blocks", "trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG
// [0.9.0]) and no CTA's first item waits on the counter.
//
// Inside a CTA the producer thread draws the indices and hands them to the
// MMA thread and the elementwise warps through a small ring in shared memory
// (full / empty mbarriers), so all roles walk the same sequence.  A cursor
// points at one stored block of one item and advances block by block.
#pragma once

#include <stdint.h>

#include "kernels.h"
#include "sm100.cuh"

namespace bsr {

constexpr int kRing = 4;

struct RingSmem {
  int32_t k[kRing];
  uint64_t full[kRing];
  uint64_t empty[kRing];
};

struct Cursor {
  int t;       // position in the CTA's item sequence
  int q;       // non-empty items started so far (per-item barrier phases)
  int g;       // blocks visited so far (per-block barrier phases)
  int i;       // block within the item
  int n;       // blocks in the item
  int line;
  int bh;
  int first;
  int slot;
  bool done;
};

struct Walk {
  const PlanItem* items;
  const PlanBucket* buckets;
  int nbuckets;
  int BH;
  int total;  // items * BH

  // Work index k -> (item, head).  Buckets of equal-length items come
  // longest first; inside a bucket the heads are the slow index and the
  // lines (ascending) the fast one, so CTAs working at the same time share a
  // head and neighbouring lines, whose K / V / Q / dO tiles overlap in L2.
  __device__ __forceinline__ void decode(int k, Cursor& c) const {
    int lo = 0, hi = nbuckets - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (buckets[mid].work <= k) lo = mid; else hi = mid - 1;
    }
    const PlanBucket b = buckets[lo];
    const int kp = k - b.work;
    const PlanItem it = items[b.start + kp % b.count];
    c.bh = kp / b.count;
    c.line = it.line;
    c.first = it.first;
    c.n = it.n;
    c.slot = it.slot;
  }

  // The same decode by a whole warp, every lane with the same k: lane i
  // reads bucket i, so a table of up to 32 buckets costs one load instead of
  // the binary search's chain of dependent loads (larger tables take
  // decode()).  The buckets ascend in their first work index and bucket 0
  // starts at 0, so the lanes whose bucket starts at or below k are 0 .. lo.
  __device__ __forceinline__ void decode_warp(int k, Cursor& c) const {
    if (nbuckets > 32) {
      decode(k, c);
      return;
    }
    const int lane = threadIdx.x % 32;
    int4 b = make_int4(0x7fffffff, 0, 1, 0);
    if (lane < nbuckets) b = *reinterpret_cast<const int4*>(buckets + lane);
    const unsigned below = __ballot_sync(0xffffffffu, b.x <= k);
    const int lo = below ? 31 - __clz(below) : 0;
    const int work = __shfl_sync(0xffffffffu, b.x, lo);
    const int start = __shfl_sync(0xffffffffu, b.y, lo);
    const int count = __shfl_sync(0xffffffffu, b.z, lo);
    const int kp = k - work;
    const PlanItem it = items[start + kp % count];
    c.bh = kp / count;
    c.line = it.line;
    c.first = it.first;
    c.n = it.n;
    c.slot = it.slot;
  }
};

__device__ __forceinline__ Walk make_walk(const PlanLayout& lay, int BH) {
  return Walk{lay.items, lay.buckets, lay.header[3], BH, lay.header[0] * BH};
}

// Warms L2 with the plan (`words` int32 from its header) before the grid
// wait, so the header, bucket table and item reads of the first draws do not
// go to HBM: lane l of the calling warp touches 128-byte line
// blockIdx.x + l * gridDim.x.  A prefetch returns no data and L2 is the point
// of coherence, so the planner may still be writing these lines; the reads
// after the grid wait see what it wrote.
__device__ __forceinline__ void plan_prefetch_l2(const int32_t* plan, size_t words) {
  const size_t line = (size_t)blockIdx.x + (size_t)(threadIdx.x % 32) * gridDim.x;
  if (line * 32 < words) asm volatile("prefetch.global.L2 [%0];" ::"l"(plan + line * 32));
}

// Producer side: draws the next work index into ring slot t % kRing once all
// consumers released it (the CTA's first draw is its block index, the later
// ones come from the counter); -1 marks the end.  Returns false on a timeout.
__device__ __forceinline__ bool ring_put(RingSmem* ring, int t, int* queue, int total, int* k_out,
                                         volatile int* abort_flag, int* status) {
  const int s = t % kRing;
  if (!sm100::mbar_wait(&ring->empty[s], ((t / kRing) & 1) ^ 1, abort_flag, status)) return false;
  int k = t == 0 ? (int)blockIdx.x : atomicAdd(queue, 1);
  if (k >= total) k = -1;
  ring->k[s] = k;
  sm100::mbar_arrive(&ring->full[s]);
  *k_out = k;
  return true;
}

// Consumer side: waits for ring slot t % kRing and returns its work index.
__device__ __forceinline__ bool ring_get(RingSmem* ring, int t, int* k_out, volatile int* abort_flag,
                                         int* status) {
  const int s = t % kRing;
  if (!sm100::mbar_wait(&ring->full[s], (t / kRing) & 1, abort_flag, status)) return false;
  *k_out = *(volatile int32_t*)&ring->k[s];
  return true;
}

__device__ __forceinline__ void ring_release(RingSmem* ring, int t) { sm100::mbar_arrive(&ring->empty[t % kRing]); }

// Sync of the 128 threads of one warpgroup on an mbarrier of count 128
// (bounded; `phase` counts the syncs this thread has done on `bar`).
__device__ __forceinline__ bool group_sync(uint64_t* bar, int& phase, volatile int* abort_flag, int* status) {
  sm100::mbar_arrive(bar);
  const bool ok = sm100::mbar_wait(bar, phase & 1, abort_flag, status);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

// Last-arriver merge of a split line.  Each chunk's warpgroup has written its
// partial result; this publishes it and tells whether this warpgroup is the
// last of the line's chunks (for this head and column half) to arrive, in
// which case it sums all the chunks' partials into the output.  `r` is the
// thread's row in the warpgroup (0..127).
__device__ __forceinline__ bool merge_arrive(const PlanLayout& lay, int slot, int bh, int BH, int hg, int r,
                                             volatile int* flag, uint64_t* bar, int& phase,
                                             volatile int* abort_flag, int* status, bool* last) {
  __threadfence();
  if (!group_sync(bar, phase, abort_flag, status)) return false;
  if (r == 0) {
    const int sl = lay.slot_line[slot];
    int* ctr = &lay.counters[(sl * BH + bh) * 2 + hg];
    const int old = atomicAdd(ctr, 1);
    const bool is_last = old == lay.line_chunks[sl] - 1;
    // the last arrival leaves the counter at 0 for the plan's next launch
    if (is_last) atomicExch(ctr, 0);
    *flag = is_last ? 1 : 0;
  }
  if (!group_sync(bar, phase, abort_flag, status)) return false;
  *last = *flag != 0;
  if (*last) __threadfence();
  return true;
}

// Called by one thread of every CTA after the CTA's last use of the plan
// (after its final __syncthreads): the last CTA of the launch to finish
// puts the work-queue counter back to the grid size and the exit count back
// to 0, so the next launch on the same plan starts from a clean queue (every
// CTA has drawn its last work index before it counts itself out).
__device__ __forceinline__ void plan_exit(const PlanLayout& lay) {
  __threadfence();
  if (atomicAdd(&lay.header[4], 1) == (int)gridDim.x - 1) {
    atomicExch(&lay.header[1], (int)gridDim.x);
    atomicExch(&lay.header[4], 0);
    __threadfence();
  }
}

// Reads 4 floats of another CTA's partial result (L2, bypassing L1).
__device__ __forceinline__ float4 ld_partial(const float* p) { return __ldcg((const float4*)p); }

// Partial tiles of split lines (fp32, 128 rows x D columns) are stored in
// groups of four columns: element (r, c) at ((c / 4) * 128 + r) * 4 + c % 4,
// so the 32 rows of a warp write and read one contiguous 512-byte run per
// group instead of 32 scattered row segments.
__device__ __forceinline__ float* part_group(float* tile, int cg, int r) { return tile + ((size_t)cg * 128 + r) * 4; }

// Stores 32 fp32 values of row r, columns [4 cg0, 4 cg0 + 32), into a tile.
__device__ __forceinline__ void part_store32(float* tile, int cg0, int r, const uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *(float4*)part_group(tile, cg0 + j, r) = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                         __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
}

// acc += w * (row r, columns [4 cg0, 4 cg0 + 32) of a tile).
__device__ __forceinline__ void part_accum32(const float* tile, int cg0, int r, float w, float (&acc)[32]) {
  float4 x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = ld_partial(part_group(const_cast<float*>(tile), cg0 + j, r));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    acc[4 * j] = fmaf(w, x[j].x, acc[4 * j]);
    acc[4 * j + 1] = fmaf(w, x[j].y, acc[4 * j + 1]);
    acc[4 * j + 2] = fmaf(w, x[j].z, acc[4 * j + 2]);
    acc[4 * j + 3] = fmaf(w, x[j].w, acc[4 * j + 3]);
  }
}

// Writes NC fp32 TMEM columns of this lane (row r) into a partial tile,
// starting at column group cg0 (see part_group).
template <int NC>
__device__ __forceinline__ void store_acc_part(uint32_t taddr, float* tile, int cg0, int r) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t v[32];
    sm100::tmem_ld32(taddr + c * 32, v);
    sm100::tmem_wait_ld();
    part_store32(tile, cg0 + c * 8, r, v);
  }
}

// Sums NC columns of row r (from column group cg0) over `nc` partial tiles
// spaced `stride` floats apart and stores them as T times `mul` at dst.
template <int NC, typename T>
__device__ __forceinline__ void merge_tiles(const float* tile0, size_t stride, int nc, int cg0, int r, T* dst,
                                            float mul) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    for (int ch = 0; ch < nc; ++ch) part_accum32(tile0 + ch * stride, cg0 + c * 8, r, 1.f, acc);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = sm100::Half16<T>::pack(acc[2 * j] * mul, acc[2 * j + 1] * mul);
    sm100::st_global_64B(dst + c * 32, w);
  }
}

}  // namespace bsr
