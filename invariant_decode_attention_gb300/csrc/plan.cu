// Split plan kernels (integer only).
//
// INVARIANT: the split count and boundaries of a row come from its own length
// and compile-time constants -- the opt-in mode proposed in "Sparse MLA decode
// is not batch-invariant" (FlashMLA issue #212, section "Question").  The
// batch enters only through the work list (which items exist and in which
// order the persistent CTAs take them); it changes where a split runs, never
// what it computes.
//
// BALANCED: the batch-wide quota of the same page's "Where it comes from"
// section -- payload = ceil(total / parts) + fixed overhead, with total summed
// over every row, then greedy packing in batch order that cuts a row wherever
// a part fills up.  The page's scheduler allows up to 256 splits; here a row
// has at most the variant's max_splits, so the quota is raised, where needed,
// to the smallest one that cuts the longest row into that many (otherwise the
// last split of a long row would take all the rest and BALANCED would be an
// unfairly slow opponent).  Kept only to measure what invariance costs.
#include "common.cuh"

namespace da {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int ceil_div_i(int a, int b) { return a / b + (a % b != 0); }

// A row's list length: its main entries plus, when a second source is given,
// its extra entries (each part clamped to its own capacity).
__device__ __forceinline__ int row_length(const PlanLaunch& p, int b) {
  const int L = p.lengths[b];
  int Lc = clamp_len(L, p.capacity);
  bool bad = Lc != L;
  if (p.extra_lengths) {
    const int Le = p.extra_lengths[b];
    const int Lec = clamp_len(Le, p.extra_capacity);
    bad |= Lec != Le;
    Lc += Lec;
  }
  if (bad) set_error(p.hdr, DA_DEVERR_LENGTH);
  return Lc;
}

__device__ __forceinline__ int row_length_quiet(const PlanLaunch& p, int b) {
  int Lc = clamp_len(p.lengths[b], p.capacity);
  if (p.extra_lengths) Lc += clamp_len(p.extra_lengths[b], p.extra_capacity);
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

// Work-list order: items with more tiles first (bucket key = tile count,
// capped at kSortKeys - 1), so that the round-robin placement of persistent
// CTAs hands out the long items before the short ones.  Placement only: an
// item's arithmetic never depends on where it lands in the list.
constexpr int kSortKeys = 256;

__device__ __forceinline__ int sort_key(int tiles) { return min(tiles, kSortKeys - 1); }

// A row's split shape under the INVARIANT rule.
struct RowSplits {
  int n, tps, n_tiles, len;
};

__device__ __forceinline__ RowSplits invariant_splits(const PlanLaunch& p, int len) {
  RowSplits r;
  r.len = len;
  r.n_tiles = ceil_div_i(len, p.tile);
  r.tps = max(p.min_tps, ceil_div_i(r.n_tiles, p.max_splits));
  r.n = max(1, ceil_div_i(r.n_tiles, r.tps));
  return r;
}

__global__ void __launch_bounds__(kPlanThreads) plan_invariant_kernel(PlanLaunch p) {
  __shared__ int bucket[kSortKeys];
  allow_next_grid();  // the split kernel may be staged now; it waits for us
  if (threadIdx.x == 0) {
    p.hdr[kHdrError] = 0;
    p.hdr[kHdrQueue] = 0;
    p.hdr[kHdrExits] = 0;
  }
  for (int k = threadIdx.x; k < kSortKeys; k += kPlanThreads) bucket[k] = 0;
  __syncthreads();
  const int stride = p.max_splits + 1;
  // pass 1: every row's splits; count items per key.  A thread keeps its
  // first row's shape in registers for pass 2.
  RowSplits mine = {0, 1, 0, 0};
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const RowSplits r = invariant_splits(p, row_length(p, b));
    if (b == (int)threadIdx.x) mine = r;
    p.n_splits[b] = r.n;
    int32_t* sb = p.split_begin + (size_t)b * stride;
    for (int s = 0; s < r.n; ++s) sb[s] = min(s * r.tps, r.n_tiles);
    sb[r.n] = r.n_tiles;
    const int last = r.n_tiles - (r.n - 1) * r.tps;  // tiles of the last split
    if (r.n > 1) atomicAdd(&bucket[sort_key(r.tps)], r.n - 1);
    atomicAdd(&bucket[sort_key(last)], 1);
  }
  __syncthreads();
  // bucket starts, largest key first: thread t < kSortKeys owns key
  // kSortKeys - 1 - t, and a block scan in that order gives the starts
  {
    static_assert(kSortKeys <= kPlanThreads, "one thread per key");
    const int key = kSortKeys - 1 - (int)threadIdx.x;
    const int count = (key >= 0) ? bucket[key] : 0;
    int total;
    const int start = block_exclusive_scan(count, &total);
    if (key >= 0) bucket[key] = start;
    if (key == 0) p.hdr[kHdrNEmpty] = count;  // items with no tiles: key 0, listed last
    if (threadIdx.x == 0) p.hdr[kHdrNWork] = total;
  }
  __syncthreads();
  // pass 2: place every item in its bucket (order within a bucket is free).
  // All splits of a row but the last have tps tiles, so a row takes n - 1
  // consecutive places of that key with one atomic and its last split one
  // place of its own key; the stores then need no further atomics.
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const RowSplits r = (b == (int)threadIdx.x) ? mine
                                                : invariant_splits(p, row_length_quiet(p, b));
    const int last0 = (r.n - 1) * r.tps;  // first tile of the last split
    const int pos_full = (r.n > 1) ? atomicAdd(&bucket[sort_key(r.tps)], r.n - 1) : 0;
    const int pos_last = atomicAdd(&bucket[sort_key(r.n_tiles - last0)], 1);
    for (int s = 0; s < r.n; ++s) {
      const int slot = b * p.max_splits + s;
      const bool is_last = s == r.n - 1;
      const int pos = is_last ? pos_last : pos_full + s;
      const int t0 = s * r.tps, t1 = is_last ? r.n_tiles : t0 + r.tps;
      p.work[pos] = slot;
      reinterpret_cast<int4*>(p.item_desc)[pos] = make_int4(r.n == 1 ? ~slot : slot, t0, t1, r.len);
    }
  }
}

// BALANCED, as the page's scheduler does it: the batch-wide total by a
// block reduction, then the greedy walk over the rows -- sequential by
// definition, each row's cuts depend on how full the current part is after
// every earlier row -- by one thread over tile counts staged in shared
// memory, then every item placed in parallel.
constexpr int kBalancedSmemRows = 8192;  // rows whose tile counts fit in shared memory

__global__ void __launch_bounds__(kPlanThreads) plan_balanced_kernel(PlanLaunch p) {
  __shared__ int bucket[kSortKeys];
  __shared__ int tiles_s[kBalancedSmemRows];
  __shared__ long long red[kPlanThreads / 32];
  __shared__ int red_max[kPlanThreads / 32];
  allow_next_grid();
  if (threadIdx.x == 0) {
    p.hdr[kHdrError] = 0;
    p.hdr[kHdrQueue] = 0;
    p.hdr[kHdrExits] = 0;
  }
  for (int k = threadIdx.x; k < kSortKeys; k += kPlanThreads) bucket[k] = 0;
  const int stride = p.max_splits + 1;
  const int ovh = p.fixed_overhead;
  const bool in_smem = p.B <= kBalancedSmemRows;
  // every row's tile count (kept in n_splits until the walk overwrites it)
  long long part = 0;
  int longest = 0;
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int n = ceil_div_i(row_length(p, b), p.tile);
    if (in_smem) tiles_s[b] = n;
    p.n_splits[b] = n;
    part += n + ovh;
    longest = max(longest, n);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    part += __shfl_xor_sync(0xffffffffu, part, o);
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = part;
    red_max[threadIdx.x >> 5] = longest;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long total = 0;
    int n_max = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      total += red[w];
      n_max = max(n_max, red_max[w]);
    }
    const int parts = max(1, p.num_parts);
    long long payload = (total / parts + (total % parts != 0)) + ovh;
    // raised, where needed, so that the longest row fits in the split budget:
    // full parts of payload - ovh tiles cut it into at most max_splits pieces
    const int cap = max(1, p.max_splits - 1);
    const long long fit = (long long)(n_max / cap + (n_max % cap != 0)) + ovh;
    if (payload < fit) payload = fit;
    long long room = payload;
    for (int b = 0; b < p.B; ++b) {
      const int n_tiles = in_smem ? tiles_s[b] : p.n_splits[b];
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
    }
  }
  __syncthreads();
  // count the items per key, then bucket starts, largest key first
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int n = p.n_splits[b];
    const int32_t* sb = p.split_begin + (size_t)b * stride;
    for (int s = 0; s < n; ++s) atomicAdd(&bucket[sort_key(sb[s + 1] - sb[s])], 1);
  }
  __syncthreads();
  {
    const int key = kSortKeys - 1 - (int)threadIdx.x;
    const int count = (key >= 0) ? bucket[key] : 0;
    int total;
    const int start = block_exclusive_scan(count, &total);
    if (key >= 0) bucket[key] = start;
    if (key == 0) p.hdr[kHdrNEmpty] = count;  // items with no tiles: key 0, listed last
    if (threadIdx.x == 0) p.hdr[kHdrNWork] = total;
  }
  __syncthreads();
  // place every item in its bucket (order within a bucket is free: placement only)
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int n = p.n_splits[b];
    const int32_t* sb = p.split_begin + (size_t)b * stride;
    const int Lc = row_length_quiet(p, b);
    for (int s = 0; s < n; ++s) {
      const int slot = b * p.max_splits + s;
      const int pos = atomicAdd(&bucket[sort_key(sb[s + 1] - sb[s])], 1);
      reinterpret_cast<int4*>(p.item_desc)[pos] =
          make_int4(n == 1 ? ~slot : slot, sb[s], sb[s + 1], Lc);
      p.work[pos] = slot;
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t stream) {
  if (p.policy == DA_POLICY_BALANCED) {
    plan_balanced_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  } else {
    plan_invariant_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace da
