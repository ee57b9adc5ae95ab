// Combine kernel: fixed-order fp32 log-sum-exp merge of the split partials of
// every (row b, query head j) whose row has n > 1 splits (the arithmetic is
// in merge.cuh).  The partial LSEs are kept in log2 units by the split
// kernel.  n depends only on the row's own length under the INVARIANT plan,
// so the addends and their order are the same in any batch.
//
// One CTA per (row, head): warp 0 forms the weights, then every thread owns up
// to four value dims (d, d + 128, ...) and advances their FMA chains together,
// split by split, so all their loads are in flight at once; each chain runs
// in split order from zero, as merge.cuh states.
#include "common.cuh"
#include "merge.cuh"

namespace da {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kMaxDimsPerThread = 4;  // D_v <= 512
constexpr int kMaxSplitsAny = kFmaMaxSplits > kMlaMaxSplits ? kFmaMaxSplits : kMlaMaxSplits;
static_assert(kMaxSplitsAny <= 64, "two split weights per lane of warp 0");

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Launch p) {
  __shared__ float coef[kMaxSplitsAny];
  __shared__ float lse_out;
  wait_prior_grid();  // the split kernel's partials
  const int b = blockIdx.x / p.H_q, j = blockIdx.x % p.H_q;
  const int n = p.n_splits[b];
  if (n <= 1) return;  // written final by the split kernel
  const size_t slot0 = (size_t)b * p.max_splits;
  if (threadIdx.x < 32) {
    const float lse = merge_weights(p.lse_part + slot0 * p.H_q + j, p.H_q, n, coef, threadIdx.x);
    if (threadIdx.x == 0) lse_out = lse;
  }
  __syncthreads();
  const int Dv = p.D_v;
  const size_t stride = (size_t)p.H_q * Dv;
  const float* o0 = p.o_part + (slot0 * p.H_q + j) * (size_t)Dv;
  float acc[kMaxDimsPerThread];
#pragma unroll
  for (int k = 0; k < kMaxDimsPerThread; ++k) acc[k] = 0.f;
#pragma unroll 2
  for (int s = 0; s < n; ++s) {
    const float c = coef[s];
#pragma unroll
    for (int k = 0; k < kMaxDimsPerThread; ++k) {
      const int d = threadIdx.x + k * kCombineThreads;
      if (d < Dv) acc[k] = fmaf(c, __ldcg(o0 + s * stride + d), acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxDimsPerThread; ++k) {
    const int d = threadIdx.x + k * kCombineThreads;
    if (d < Dv) p.out[((size_t)b * p.H_q + j) * Dv + d] = __float2bfloat16_rn(acc[k]);
  }
  if (threadIdx.x == 0) p.lse[(size_t)b * p.H_q + j] = lse_out;
}

}  // namespace

cudaError_t launch_combine(const Launch& p, cudaStream_t stream) {
  if (p.D_v > kCombineThreads * kMaxDimsPerThread) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.B * p.H_q;
  if (blocks == 0) return cudaSuccess;
  return launch_after(combine_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, p);
}

}  // namespace da
