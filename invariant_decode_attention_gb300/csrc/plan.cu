// Split plan kernels (integer only).
//
// INVARIANT: the split count and boundaries of a row come from its own length
// and compile-time constants -- the opt-in mode proposed in "Sparse MLA decode
// is not batch-invariant" (FlashMLA issue #212, section "Question").  The
// batch enters only through the work list (a prefix sum that places items; it
// changes where a split runs, never what it computes).
//
// BALANCED: the batch-wide quota of the same page's "Where it comes from"
// section -- payload = ceil(total / parts) + fixed overhead, with total summed
// over every row, then greedy packing in batch order that cuts a row wherever
// a part fills up.  Kept only to measure what invariance costs.
#include "common.cuh"

namespace da {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int ceil_div_i(int a, int b) { return a / b + (a % b != 0); }

__device__ __forceinline__ int row_length(const PlanLaunch& p, int b) {
  const int L = p.lengths[b];
  const int Lc = clamp_len(L, p.capacity);
  if (Lc != L) set_error(p.hdr, DA_DEVERR_LENGTH);
  return Lc;
}

// Exclusive block-wide prefix sum of one int per thread; also returns the total.
__device__ int block_exclusive_scan(int x, int* total) {
  __shared__ int warp_sums[kPlanThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int warp_base = warp == 0 ? 0 : warp_sums[warp - 1];
  *total = warp_sums[kPlanThreads / 32 - 1];
  __syncthreads();
  return warp_base + incl - x;
}

__global__ void __launch_bounds__(kPlanThreads) plan_invariant_kernel(PlanLaunch p) {
  if (threadIdx.x == 0) p.hdr[kHdrError] = 0;
  __syncthreads();
  const int stride = p.max_splits + 1;
  int work_base = 0;
  for (int base = 0; base < p.B; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    int n = 0, n_tiles = 0, tps = 1;
    if (b < p.B) {
      const int L = row_length(p, b);
      n_tiles = ceil_div_i(L, p.tile);
      tps = max(p.min_tps, ceil_div_i(n_tiles, p.max_splits));
      n = max(1, ceil_div_i(n_tiles, tps));
      p.n_splits[b] = n;
      int32_t* sb = p.split_begin + (size_t)b * stride;
      for (int s = 0; s < n; ++s) sb[s] = min(s * tps, n_tiles);
      sb[n] = n_tiles;
    }
    int total;
    const int off = block_exclusive_scan(n, &total);
    const int Lc = (b < p.B) ? clamp_len(p.lengths[b], p.capacity) : 0;
    for (int s = 0; s < n; ++s) {
      const int slot = b * p.max_splits + s;
      p.work[work_base + off + s] = slot;
      reinterpret_cast<int4*>(p.item_desc)[work_base + off + s] =
          make_int4(n == 1 ? ~slot : slot, min(s * tps, n_tiles), min((s + 1) * tps, n_tiles), Lc);
    }
    work_base += total;
  }
  if (threadIdx.x == 0) p.hdr[kHdrNWork] = work_base;
}

// One thread: the packing is sequential by definition (each row's cuts depend
// on how full the current part is after every earlier row).
__global__ void plan_balanced_kernel(PlanLaunch p) {
  if (threadIdx.x != 0) return;
  p.hdr[kHdrError] = 0;
  const int stride = p.max_splits + 1;
  const int ovh = p.fixed_overhead;
  long long total = 0;
  for (int b = 0; b < p.B; ++b) total += ceil_div_i(row_length(p, b), p.tile) + ovh;
  const int parts = max(1, p.num_parts);
  const long long payload = (total / parts + (total % parts != 0)) + ovh;
  long long room = payload;
  int n_work = 0;
  for (int b = 0; b < p.B; ++b) {
    const int n_tiles = ceil_div_i(clamp_len(p.lengths[b], p.capacity), p.tile);
    int32_t* sb = p.split_begin + (size_t)b * stride;
    int n_cuts = 1;  // entries written to sb so far
    sb[0] = 0;
    long long begin = 0;
    for (;;) {
      const long long rest = n_tiles - begin;
      if (rest + ovh <= room) {  // the rest of the row fits in this part
        room -= rest + ovh;
        break;
      }
      const long long take = room - ovh;
      if (take > 0 && n_cuts < p.max_splits) {  // fill the part, cut the row
        begin += take;
        sb[n_cuts++] = (int)begin;
      }
      room = payload;  // open a new part
      if (n_cuts == p.max_splits) {  // no splits left: the last one takes the rest
        room = room - (n_tiles - begin) - ovh;
        if (room < 0) room = 0;
        break;
      }
    }
    sb[n_cuts] = n_tiles;
    p.n_splits[b] = n_cuts;
    const int Lc = clamp_len(p.lengths[b], p.capacity);
    for (int s = 0; s < n_cuts; ++s) {
      const int slot = b * p.max_splits + s;
      reinterpret_cast<int4*>(p.item_desc)[n_work] =
          make_int4(n_cuts == 1 ? ~slot : slot, sb[s], sb[s + 1], Lc);
      p.work[n_work++] = slot;
    }
  }
  p.hdr[kHdrNWork] = n_work;
}

}  // namespace

cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t stream) {
  if (p.policy == DA_POLICY_BALANCED) {
    plan_balanced_kernel<<<1, 32, 0, stream>>>(p);
  } else {
    plan_invariant_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace da
