// Work lists for the persistent attention kernels.
//
// For each list (block rows for the forward and dQ walks, block columns for
// the dK/dV walk) the planner
//   * splits every line longer than L stored blocks into ceil(len / L)
//     chunks of nearly equal length, L = max(8, ceil(nnzb * BH / G)) (G =
//     persistent CTAs), so that no single item is longer than the average
//     share of one CTA;
//   * sorts the items by length, longest first, lines ascending inside a
//     length (a counting sort; the order changes the schedule, never a
//     result), and records one bucket per length; the kernels read work
//     index k of a bucket as head k / count, item k % count of the bucket
//     (see sched.cuh);
//   * leaves out lines with no stored block when asked (skip_empty; their
//     outputs are written by a separate pass), so that no persistent CTA
//     draws a run of empty items;
//   * gives each chunk of a split line a partial-result slot, and zeroes the
//     per-(line, head, column half) arrival counters used by the last-arriver
//     merge, and sets the work-queue counter to the grid size (CTA b takes
//     work index b first without it, see sched.cuh).
// Balancing the work by stored blocks with one writer per output tile
// follows "trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.9.0].
// Plan layout (int32): see PlanLayout in kernels.h.

#include "delta.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace bsr {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int line_len(const int32_t* ptr, int i, int n) {
  int c = ptr[i + 1] - ptr[i];
  return c < 0 ? 0 : (c > n ? n : c);
}

// Block-wide exclusive scan of hist[0..n] taken from the top value down:
// afterwards hist[v] = number of items with length > v.
__device__ void scan_desc(int* hist, int n, int* warp_sums) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int len = n + 1;
  const int seg = (len + nt - 1) / nt;
  // thread tid owns reversed positions [tid * seg, tid * seg + seg): values n - p
  int local = 0;
  for (int p = tid * seg; p < tid * seg + seg && p < len; ++p) local += hist[n - p];
  // inclusive warp scan of the per-thread sums
  const int lane = tid % 32, w = tid / 32;
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int v = lane < nt / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_sums[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  int run = x - local + (w > 0 ? warp_sums[w - 1] : 0);  // exclusive prefix of this thread
  for (int p = tid * seg; p < tid * seg + seg && p < len; ++p) {
    const int h = hist[n - p];
    hist[n - p] = run;
    run += h;
  }
  __syncthreads();
}

// Chunking of a line of `len` blocks when no chunk may exceed Lmax: nc
// chunks, the first r of length b + 1 and the others of length b.  Returned
// as b, and r << 16 | nc (nc <= len / 8 + 1 < 2^16 for the lists the
// planner accepts).
__device__ __forceinline__ int chunking(int len, int Lmax, int* rn) {
  const int nc = len > Lmax ? (len + Lmax - 1) / Lmax : 1;
  *rn = ((len % nc) << 16) | nc;
  return len / nc;
}

// Shared-memory ints plan_body needs for n lines: hist, count, bucket rank
// and the prefix offsets ([n + 1] each), chunk length b, r << 16 | nc and
// first block offset ([n] each).
__host__ __device__ constexpr size_t plan_smem_ints(int n) { return 4 * ((size_t)n + 1) + 3 * (size_t)n; }

// Builds list `li` of p with the whole CTA in sm_plan (plan_smem_ints(n)).
__device__ void plan_body(const PlanArgs& p, int li, int* sm_plan) {
  __shared__ int warp_sums[32];
  __shared__ int counts[3];         // items, split lines, slots
  const PlanList& L = p.list[li];
  const int n = p.n;
  int* hist = sm_plan;
  int* count = sm_plan + (n + 1);
  int* rank = sm_plan + 2 * (n + 1);
  int* ptr = sm_plan + 3 * (n + 1);  // the list's prefix offsets, staged once
  int* cb = sm_plan + 4 * (n + 1);
  int* crn = cb + n;
  int* offs = crn + n;
  PlanLayout lay = plan_layout(L.plan, n, p.G, p.BH, p.max_len);

  // all offsets in one round trip to memory
  for (int v = threadIdx.x; v <= n; v += blockDim.x) {
    hist[v] = 0;
    ptr[v] = L.ptr[v];
  }
  if (threadIdx.x < 3) counts[threadIdx.x] = 0;
  __syncthreads();

  const long long nnzb = ptr[n] > 0 ? ptr[n] : 0;
  long long lim = (nnzb * p.BH + p.G - 1) / p.G;
  if (lim < 8) lim = 8;
  // chunks never exceed n blocks (the histograms are indexed by length
  // 0..n; a square grid has no longer line, so without allow_split nothing
  // is cut)
  const int Lmax = p.allow_split ? (int)(lim < n ? lim : n) : n;
  const int max_len = p.max_len > 0 ? p.max_len : n;

  // pass 1: chunking of every line and histogram of chunk lengths
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int len = line_len(ptr, i, max_len);
    offs[i] = ptr[i];
    if (len == 0 && p.skip_empty) {  // no item: no chunk of any length
      cb[i] = 0;
      crn[i] = 0;
      continue;
    }
    int rn;
    const int bl = chunking(len, Lmax, &rn);
    cb[i] = bl;
    crn[i] = rn;
    const int nc = rn & 0xFFFF, r = rn >> 16;
    if (r > 0) atomicAdd(&hist[bl + 1], r);
    atomicAdd(&hist[bl], nc - r);
    atomicAdd(&counts[0], nc);
  }
  __syncthreads();
  for (int v = threadIdx.x; v <= n; v += blockDim.x) {
    count[v] = hist[v];
    rank[v] = hist[v] > 0 ? 1 : 0;
  }
  __syncthreads();
  scan_desc(hist, n, warp_sums);  // hist[v] = first item of length v
  scan_desc(rank, n, warp_sums);  // rank[v] = bucket of length v (longest first)
  // bucket table
  for (int v = threadIdx.x; v <= n; v += blockDim.x)
    if (count[v] > 0) lay.buckets[rank[v]] = PlanBucket{hist[v] * p.BH, hist[v], count[v], v};
  if (threadIdx.x == 0) lay.header[3] = rank[0] + (count[0] > 0 ? 1 : 0);

  // pass 2: place the items; inside a length bucket lines ascend (stable),
  // so CTAs that start together work on neighbouring lines
  const bool stable = n <= 2048;  // O(n^2 / threads) shared-memory reads
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int bl = cb[i], nc = crn[i] & 0xFFFF, rl = crn[i] >> 16;
    int base = -1;
    if (nc > 1) {
      const int sl = atomicAdd(&counts[1], 1);
      base = atomicAdd(&counts[2], nc);
      if (sl < lay.cap_lines && base + nc <= lay.cap_slots) {
        lay.line_base[sl] = base;
        lay.line_chunks[sl] = nc;
        for (int c = 0; c < nc; ++c) lay.slot_line[base + c] = sl;
      } else {
        atomicExch(p.status, kStatusDeviceCheck);
        base = -1;
      }
    }
    // items of length bl + 1 and bl of the lines before this one
    int before_hi = 0, before_lo = 0;
    if (stable) {
      for (int j = 0; j < i; ++j) {
        const int bj = cb[j], ncj = crn[j] & 0xFFFF, rj = crn[j] >> 16;
        before_hi += (bj + 1 == bl + 1 ? rj : 0) + (bj == bl + 1 ? ncj - rj : 0);
        before_lo += (bj + 1 == bl ? rj : 0) + (bj == bl ? ncj - rj : 0);
      }
    }
    int off = offs[i];
    for (int c = 0; c < nc; ++c) {
      const bool hi = c < rl;
      const int clen = bl + (hi ? 1 : 0);
      int pos;
      if (stable) {
        pos = hist[clen] + (hi ? before_hi + c : before_lo + (c - rl));
      } else {
        pos = atomicAdd(&hist[clen], 1);
      }
      if (pos < lay.cap_items) lay.items[pos] = PlanItem{i, off, clen, base < 0 ? -1 : base + c};
      off += clen;
    }
  }
  __syncthreads();
  const int nsl = counts[1] < lay.cap_lines ? counts[1] : lay.cap_lines;
  for (int x = threadIdx.x; x < nsl * p.BH * 2; x += blockDim.x) lay.counters[x] = 0;
  if (threadIdx.x == 0) {
    const int items = counts[0] <= lay.cap_items ? counts[0] : 0;
    if (counts[0] > lay.cap_items) atomicExch(p.status, kStatusDeviceCheck);
    lay.header[0] = items;
    lay.header[1] = p.G;  // work-queue counter: indices below G go to CTAs by block index
    lay.header[2] = nsl;
    lay.header[4] = 0;  // CTAs finished
    lay.header[5] = lay.header[6] = lay.header[7] = 0;
  }
}

// CTAs [0, lists) build one plan each; the p.zero_ctas CTAs after them
// write the outputs of the empty lines (zero_lines_body).
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs p, int lists) {
  sm100::griddep_wait();  // may run as a programmatic dependent
  sm100::griddep_launch_dependents();
  extern __shared__ int sm_plan[];
  if ((int)blockIdx.x < lists)
    plan_body(p, blockIdx.x, sm_plan);
  else
    zero_lines_body(p.zero, (int)blockIdx.x - lists, (int)gridDim.x - lists);
}

// Delta / lse2 of the backward pass and its work lists in one launch: the
// first `lists` CTAs build the plans, the next p.zero_ctas write the outputs
// of the empty lines, and the others compute the per-row statistics (the
// three are independent; all must be done before dQ and dK / dV start).
constexpr int kFusedThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kFusedThreads) delta_plan_kernel(BwdArgs a, PlanArgs p, int lists) {
  sm100::griddep_wait();  // may run as a programmatic dependent
  sm100::griddep_launch_dependents();
  extern __shared__ int sm_plan[];
  const int b = (int)blockIdx.x, zc = p.zero_ctas;
  if (b < lists)
    plan_body(p, b, sm_plan);
  else if (b < lists + zc)
    zero_lines_body(p.zero, b - lists, zc);
  else
    delta_pass<T, D, kFusedThreads>(a, b - lists - zc, (int)gridDim.x - lists - zc);
}

template <typename T, int D>
bsr_status launch_fused(const BwdArgs& a, const PlanArgs& p, int lists, size_t smem, cudaStream_t s) {
  const size_t rows = (size_t)a.d.BH * a.d.S;
  constexpr size_t per = delta_rows_per_cta<T, D, kFusedThreads>();
  const size_t groups = (rows + per - 1) / per;
  // one delta CTA per row group (DeltaShape, delta.cuh)
  const unsigned grid = (unsigned)(lists + p.zero_ctas + groups);
  LaunchTimer timer("delta_plan", s);
  const cudaError_t e = launch_dependent(delta_plan_kernel<T, D>, dim3(grid), dim3(kFusedThreads), smem, s, a, p, lists);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "delta_plan launch: %s", cudaGetErrorString(e));
  return check_launch("delta_plan launch");
}

}  // namespace

// The screened SpMM's tile list, then its plan, in one CTA.
__device__ __forceinline__ int tile_class(float2 row, float2 col, float t) {
  if (!(row.y * col.y > t)) return kTileSkip;
  return row.x * col.x > t ? kTileFull : kTilePartial;
}

__global__ void __launch_bounds__(kPlanThreads) screen_plan_kernel(ScreenListArgs s, PlanArgs p) {
  sm100::griddep_wait();  // may run as a programmatic dependent
  sm100::griddep_launch_dependents();
  __shared__ float2 bnd[kScreenMaxBlocks];
  __shared__ int cnt[kScreenMaxBlocks + 1];
  extern __shared__ int sm_plan[];
  const int lane = threadIdx.x % 32, wp = threadIdx.x / 32, nw = blockDim.x / 32;
  // bounds of every 128-block: one warp per block, 4 values per lane
  for (int k = wp; k < s.nb; k += nw) {
    const float4 x = ((const float4*)(s.diag + (size_t)k * 128))[lane];
    const float q0 = sqrtf(fabsf(x.x)), q1 = sqrtf(fabsf(x.y)), q2 = sqrtf(fabsf(x.z)), q3 = sqrtf(fabsf(x.w));
    float lo = fminf(fminf(q0, q1), fminf(q2, q3)), hi = fmaxf(fmaxf(q0, q1), fmaxf(q2, q3));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) bnd[k] = make_float2(lo, hi);
  }
  __syncthreads();
  // kept tiles per block row (one warp per row)
  for (int m = wp; m < s.nb; m += nw) {
    int c = 0;
    for (int k0 = 0; k0 < s.nb; k0 += 32) {
      const int k = k0 + lane;
      const bool kept = k < s.nb && tile_class(bnd[m], bnd[k], s.t) != kTileSkip;
      c += __popc(__ballot_sync(0xffffffffu, kept));
    }
    if (lane == 0) cnt[m] = c;
  }
  __syncthreads();
  if (wp == 0) {  // exclusive prefix sum of the counts by one warp
    int run = 0;
    for (int m0 = 0; m0 < s.nb; m0 += 32) {
      const int m = m0 + lane;
      const int c = m < s.nb ? cnt[m] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (m < s.nb) {
        cnt[m] = run + x - c;
        s.row_ptr[m] = run + x - c;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s.row_ptr[s.nb] = run;
  }
  __syncthreads();
  for (int m = wp; m < s.nb; m += nw) {
    int off = cnt[m];
    for (int k0 = 0; k0 < s.nb; k0 += 32) {
      const int k = k0 + lane;
      const int cl = k < s.nb ? tile_class(bnd[m], bnd[k], s.t) : kTileSkip;
      const unsigned kept = __ballot_sync(0xffffffffu, cl != kTileSkip);
      if (cl != kTileSkip) {
        const int pos = off + __popc(kept & ((1u << lane) - 1u));
        s.col_idx[pos] = k;
        s.cls[pos] = cl;
      }
      off += __popc(kept);
    }
  }
  // the list is in global memory, written by this CTA: the plan reads it back
  __threadfence_block();
  __syncthreads();
  plan_body(p, 0, sm_plan);
}

// Planner threads: enough for one line each (the loops stride past that),
// a whole number of warps, at most the kernel's bound.
static int plan_threads(int n) {
  const int t = ((n + 1 + 31) / 32) * 32;
  return t < 128 ? 128 : (t > kPlanThreads ? kPlanThreads : t);
}

bsr_status launch_plan(const PlanArgs& p, int lists, cudaStream_t s) {
  const size_t smem = sizeof(int) * plan_smem_ints(p.n);
  if (smem > 200 * 1024) return fail(BSR_ERR_UNSUPPORTED, "plan: %d block rows exceed the planner's limit", p.n);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "plan: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  LaunchTimer timer("plan", s);
  const cudaError_t e =
      launch_dependent(plan_kernel, dim3(lists + p.zero_ctas), dim3(plan_threads(p.n)), smem, s, p, lists);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "plan launch: %s", cudaGetErrorString(e));
  return check_launch("plan launch");
}

bsr_status launch_screen_plan(const ScreenListArgs& l, const PlanArgs& p, cudaStream_t s) {
  if (l.nb < 1 || l.nb > kScreenMaxBlocks || p.n != l.nb)
    return fail(BSR_ERR_UNSUPPORTED, "screened list: %d block rows (1 .. %d)", l.nb, (int)kScreenMaxBlocks);
  const size_t smem = sizeof(int) * plan_smem_ints(p.n);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(screen_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "screen_plan: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  LaunchTimer timer("screen_plan", s);
  const cudaError_t e = launch_dependent(screen_plan_kernel, dim3(1), dim3(kPlanThreads), smem, s, l, p);
  if (e != cudaSuccess) return fail(BSR_ERR_CUDA, "screen_plan launch: %s", cudaGetErrorString(e));
  return check_launch("screen_plan launch");
}

bsr_status launch_delta_plan(const BwdArgs& a, const PlanArgs& p, int lists, cudaStream_t s) {
  // fused only while the planner's shared memory and its O(n^2 / threads)
  // stable placement stay small
  const size_t smem = sizeof(int) * plan_smem_ints(p.n);
  const bool fuse = p.n <= 512 && a.d.dtype != BSR_F32 && (a.d.D == 64 || a.d.D == 128);
  if (!fuse) {
    bsr_status st = launch_delta(a, s);
    if (st != BSR_OK) return st;
    return launch_plan(p, lists, s);
  }
  if (a.d.dtype == BSR_F16)
    return a.d.D == 64 ? launch_fused<__half, 64>(a, p, lists, smem, s) : launch_fused<__half, 128>(a, p, lists, smem, s);
  return a.d.D == 64 ? launch_fused<__nv_bfloat16, 64>(a, p, lists, smem, s)
                     : launch_fused<__nv_bfloat16, 128>(a, p, lists, smem, s);
}

}  // namespace bsr
