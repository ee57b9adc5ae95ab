// Combine kernel: fixed-order fp32 log-sum-exp merge of the split partials of
// every (row b, query head j) whose row has n > 1 splits (the arithmetic is
// in merge.cuh).  The partial LSEs are kept in log2 units by the split
// kernel.  n depends only on the row's own length under the INVARIANT plan,
// so the addends and their order are the same in any batch.
//
// One CTA per (row, head): every thread owns up to four value dims (d,
// d + 128, ...).  It loads its values of a batch of NB splits first (all
// those loads in flight at once; the first batch is issued before warp 0
// forms the weights), then advances its FMA chains through the batch; each
// chain runs in split order from zero, as merge.cuh states.  NB is the
// bound on any row's split count that the plan implies (16 or 64 for one
// value dim per thread), so a row costs one round trip to L2 without holding
// registers for splits no row can have.  Rows of at most 16 splits with
// D_v <= 128 take combine_warp_kernel instead: one warp per (row, head),
// a lane per four value dims, so a split's values are one 16-byte load per
// lane and four heads share a CTA.
#include "common.cuh"
#include "merge.cuh"

namespace da {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kMaxDimsPerThread = 4;  // D_v <= 512
constexpr int kMaxSplitsAny = kFmaMaxSplits > kMlaMaxSplits ? kFmaMaxSplits : kMlaMaxSplits;
static_assert(kMaxSplitsAny <= 64, "two split weights per lane of warp 0");

// DPT: value dims per thread (1 when D_v <= 128, else up to 4); NB: splits
// whose loads are issued together.
template <int DPT, int NB>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Launch p) {
  __shared__ float coef[kMaxSplitsAny];
  __shared__ float lse_out;
  wait_prior_grid();  // the split kernel's partials
  const int b = blockIdx.x / p.H_q, j = blockIdx.x % p.H_q;
  const int n = p.n_splits[b];
  if (n <= 1) return;  // written final by the split kernel
  const size_t slot0 = (size_t)b * p.max_splits;
  const int Dv = p.D_v;
  const size_t stride = (size_t)p.H_q * Dv;
  const float* o0 = p.o_part + (slot0 * p.H_q + j) * (size_t)Dv + threadIdx.x;
  const int nk = (Dv - (int)threadIdx.x + kCombineThreads - 1) / kCombineThreads;  // own dims
  float v[NB][DPT];
  auto load = [&](int s0) {
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
      for (int k = 0; k < DPT; ++k)
        v[i][k] = (s0 + i < n && k < nk)
                      ? __ldcg(o0 + (size_t)(s0 + i) * stride + k * kCombineThreads)
                      : 0.f;
  };
  load(0);  // in flight while warp 0 forms the weights
  if (threadIdx.x < 32) {
    const float lse = merge_weights(p.lse_part + slot0 * p.H_q + j, p.H_q, n, coef, threadIdx.x);
    if (threadIdx.x == 0) lse_out = lse;
  }
  __syncthreads();
  float acc[DPT];
#pragma unroll
  for (int k = 0; k < DPT; ++k) acc[k] = 0.f;
  for (int s0 = 0; s0 < n; s0 += NB) {
    if (s0 > 0) load(s0);
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      if (s0 + i < n) {
        const float c = coef[s0 + i];
#pragma unroll
        for (int k = 0; k < DPT; ++k) acc[k] = fmaf(c, v[i][k], acc[k]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < DPT; ++k) {
    const int d = threadIdx.x + k * kCombineThreads;
    if (d < Dv) p.out[((size_t)b * p.H_q + j) * Dv + d] = __float2bfloat16_rn(acc[k]);
  }
  if (threadIdx.x == 0) p.lse[(size_t)b * p.H_q + j] = lse_out;
}

// One warp per (row, head), for D_v <= 128 and rows of at most NB splits
// (the plan's bound): lane l owns value dims 4l .. 4l + 3, so one 16-byte
// load per lane takes a split's whole row of values for the head, and the
// loads of every split are in flight while the warp forms the weights.  Per
// value dim the FMA chain is combine_kernel's: split order from zero.  (A
// row with more than NB splits, which the plan rules out, would still be
// merged in order by the loop after the batch.)
constexpr int kCombineWarps = kCombineThreads / 32;

template <int NB>
__global__ void __launch_bounds__(kCombineThreads) combine_warp_kernel(Launch p) {
  __shared__ float coef[kCombineWarps][kMaxSplitsAny];
  wait_prior_grid();  // the split kernel's partials
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kCombineWarps + warp;
  if (item >= (long long)p.B * p.H_q) return;
  const int b = (int)(item / p.H_q), j = (int)(item % p.H_q);
  const int n = p.n_splits[b];
  if (n <= 1) return;  // written final by the split kernel
  const size_t slot0 = (size_t)b * p.max_splits;
  const int Dv = p.D_v;
  const bool mine = 4 * lane < Dv;
  const size_t stride4 = (size_t)p.H_q * Dv / 4;  // float4s per split
  const float4* o0 = reinterpret_cast<const float4*>(p.o_part + (slot0 * p.H_q + j) * Dv) + lane;
  float4 v[NB];
#pragma unroll
  for (int s = 0; s < NB; ++s)
    v[s] = (s < n && mine) ? __ldcg(o0 + (size_t)s * stride4) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float lse = merge_weights(p.lse_part + slot0 * p.H_q + j, p.H_q, n, coef[warp], lane);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fma4 = [&](float c, const float4& x) {
    acc.x = fmaf(c, x.x, acc.x);
    acc.y = fmaf(c, x.y, acc.y);
    acc.z = fmaf(c, x.z, acc.z);
    acc.w = fmaf(c, x.w, acc.w);
  };
#pragma unroll
  for (int s = 0; s < NB; ++s)
    if (s < n) fma4(coef[warp][s], v[s]);
  for (int s = NB; s < n; ++s)
    fma4(coef[warp][s], mine ? __ldcg(o0 + (size_t)s * stride4) : make_float4(0.f, 0.f, 0.f, 0.f));
  if (mine) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    *reinterpret_cast<uint2*>(p.out + ((size_t)b * p.H_q + j) * Dv + 4 * lane) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
  if (lane == 0) p.lse[(size_t)b * p.H_q + j] = lse;
}

// The tensor-core variant's partials are head-interleaved: value dims in
// groups of four, heads innermost -- element (slot, head j, dim d) at
// ((slot * 128 + d / 4) * H_q + j) * 4 + d % 4 -- so that its epilogue's
// stores coalesce.  Its combine takes one thread per (row, head, four 4-dim
// groups): a warp's load of one split's group covers 32 consecutive heads
// (512 contiguous bytes).  Every thread forms its head's weights itself with
// the operations and order of merge_weights (its LSEs staged in its own
// shared-memory column), and the loads of a whole batch of splits, together
// with the split LSEs, are in flight at once: a row with up to kMlaBatch
// splits costs one round trip to L2.
constexpr int kMlaThreads = 128;
constexpr int kMlaGroupsPerThread = 4;  // 4-dim groups: 16 value dims, one 32-byte sector of out
constexpr int kMlaGroupsPerCta = (kMlaThreads / 128) * kMlaGroupsPerThread;
constexpr int kMlaBatch = 4;  // splits whose loads are issued together

__global__ void __launch_bounds__(kMlaThreads) combine_mla_kernel(Launch p) {
  __shared__ float col[kMlaMaxSplits][kMlaThreads];  // thread t's column: its LSEs, then weights
  wait_prior_grid();  // the split kernel's partials
  constexpr int kCtasPerRow = 512 / 4 / kMlaGroupsPerCta;
  const int b = blockIdx.x / kCtasPerRow, cb = blockIdx.x % kCtasPerRow;
  const int n = p.n_splits[b];
  const int t = threadIdx.x, j = t & 127;
  if (n <= 1 || j >= p.H_q) return;
  const int g0 = cb * kMlaGroupsPerCta + (t >> 7) * kMlaGroupsPerThread;
  const size_t slot0 = (size_t)b * p.max_splits;
  const size_t split_stride = (size_t)128 * p.H_q;  // float4s per split
  const float4* base = reinterpret_cast<const float4*>(p.o_part) + (slot0 * 128 + g0) * p.H_q + j;
  float4 v[kMlaBatch][kMlaGroupsPerThread];
  auto load = [&](int s0) {
#pragma unroll
    for (int i = 0; i < kMlaBatch; ++i)
#pragma unroll
      for (int e = 0; e < kMlaGroupsPerThread; ++e)
        v[i][e] = (s0 + i < n) ? __ldcg(base + (size_t)(s0 + i) * split_stride + e * p.H_q)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  load(0);  // in flight with the LSE loads
  // weights: M = max of the split LSEs, w_s = 2^(lse_s - M), W = sum in
  // split order, coefficient w_s / W (merge_weights' arithmetic)
  const float* lse = p.lse_part + slot0 * p.H_q + j;
  float M = -INFINITY;
  for (int s0 = 0; s0 < n; s0 += 8) {
    float ls[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ls[i] = (s0 + i < n) ? __ldcg(lse + (size_t)(s0 + i) * p.H_q) : -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (s0 + i < n) col[s0 + i][t] = ls[i];
      M = fmaxf(M, ls[i]);
    }
  }
  float W = 0.f;
  for (int s = 0; s < n; ++s) {
    const float w = (M == -INFINITY) ? 0.f : ex2(col[s][t] - M);
    col[s][t] = w;
    W += w;
  }
  for (int s = 0; s < n; ++s) col[s][t] = (W > 0.f) ? col[s][t] / W : 0.f;
  float4 acc[kMlaGroupsPerThread];
#pragma unroll
  for (int e = 0; e < kMlaGroupsPerThread; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += kMlaBatch) {
    if (s0 > 0) load(s0);
#pragma unroll
    for (int i = 0; i < kMlaBatch; ++i) {
      if (s0 + i < n) {
        const float c = col[s0 + i][t];
#pragma unroll
        for (int e = 0; e < kMlaGroupsPerThread; ++e) {
          acc[e].x = fmaf(c, v[i][e].x, acc[e].x);
          acc[e].y = fmaf(c, v[i][e].y, acc[e].y);
          acc[e].z = fmaf(c, v[i][e].z, acc[e].z);
          acc[e].w = fmaf(c, v[i][e].w, acc[e].w);
        }
      }
    }
  }
  uint32_t w[2 * kMlaGroupsPerThread];
#pragma unroll
  for (int e = 0; e < kMlaGroupsPerThread; ++e) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[e].x, acc[e].y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[e].z, acc[e].w);
    w[2 * e] = *reinterpret_cast<const uint32_t*>(&lo);
    w[2 * e + 1] = *reinterpret_cast<const uint32_t*>(&hi);
  }
  uint4* dsto = reinterpret_cast<uint4*>(p.out + ((size_t)b * p.H_q + j) * 512 + g0 * 4);
  dsto[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dsto[1] = make_uint4(w[4], w[5], w[6], w[7]);
  if (cb == 0 && t < 128) p.lse[(size_t)b * p.H_q + j] = (W > 0.f) ? (M + lg2(W)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Launch& p, int n_bound, cudaStream_t stream) {
  if (p.o_part_mla) {
    if (p.D_v != 512 || p.H_q > 128) return cudaErrorInvalidValue;
    const long long blocks = (long long)p.B * (512 / 4 / kMlaGroupsPerCta);
    if (blocks == 0) return cudaSuccess;
    return launch_after(combine_mla_kernel, dim3((unsigned)blocks), dim3(kMlaThreads), 0, stream,
                        p);
  }
  if (p.D_v > kCombineThreads * kMaxDimsPerThread) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.B * p.H_q;
  if (blocks == 0) return cudaSuccess;
  if (p.D_v <= kCombineThreads && p.D_v % 4 == 0 && n_bound <= 16) {
    const long long warp_blocks = (blocks + kCombineWarps - 1) / kCombineWarps;
    if (n_bound <= 8)
      return launch_after(combine_warp_kernel<8>, dim3((unsigned)warp_blocks),
                          dim3(kCombineThreads), 0, stream, p);
    return launch_after(combine_warp_kernel<16>, dim3((unsigned)warp_blocks),
                        dim3(kCombineThreads), 0, stream, p);
  }
  if (p.D_v <= kCombineThreads) {
    if (n_bound <= 16)
      return launch_after(combine_kernel<1, 16>, dim3((unsigned)blocks), dim3(kCombineThreads), 0,
                          stream, p);
    return launch_after(combine_kernel<1, 64>, dim3((unsigned)blocks), dim3(kCombineThreads), 0,
                        stream, p);
  }
  return launch_after(combine_kernel<kMaxDimsPerThread, 16>, dim3((unsigned)blocks),
                      dim3(kCombineThreads), 0, stream, p);
}

cudaError_t launch_combine(const Launch& p, cudaStream_t stream) {
  return launch_combine(p, p.max_splits, stream);
}

}  // namespace da
