// Combine kernel: fixed-order fp32 log-sum-exp merge of a row's split partials.
//
// For every (row b, query head j) whose row has n > 1 splits:
//     M   = max_s lse_s                       (exact; order-free)
//     w_s = 2^(lse_s - M),  W = w_0 + w_1 + ... + w_{n-1}   (in this order)
//     out = sum_s (w_s / W) * o_s             (fp32, s = 0 .. n-1 in order)
//     lse = (M + log2 W) * ln 2               (natural log)
// The partial LSEs are kept in log2 units by the split kernel.  n depends only
// on the row's own length under the INVARIANT plan, so the addends and their
// order are the same in any batch.  The merge is the combine step of FlashMLA
// issue #212 ("Where it comes from": the per-split LSE rescale followed by a
// sequential fp32 sum), with its split count taken from the per-row plan.
//
// One CTA per (row, head): warp 0 forms the weights, then every thread owns
// value dims and walks the splits in order with several loads in flight.
#include "common.cuh"

namespace da {
namespace {

constexpr int kCombineThreads = 128;
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
    const int lane = threadIdx.x;
    float ls[2];
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int s = lane + 32 * i;
      ls[i] = (s < n) ? p.lse_part[(slot0 + s) * p.H_q + j] : -INFINITY;
      M = fmaxf(M, ls[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int s = lane + 32 * i;
      if (s < n) coef[s] = (M == -INFINITY) ? 0.f : ex2(ls[i] - M);
    }
    __syncwarp();
    float W = 0.f;
    for (int s = 0; s < n; ++s) W += coef[s];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int s = lane + 32 * i;
      if (s < n) coef[s] = (W > 0.f) ? coef[s] / W : 0.f;
    }
    if (lane == 0) lse_out = (W > 0.f) ? (M + lg2(W)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  const int Dv = p.D_v;
  const size_t slot_stride = (size_t)p.H_q * Dv;
  const float* o0 = p.o_part + (slot0 * p.H_q + j) * (size_t)Dv;
  for (int d = threadIdx.x; d < Dv; d += kCombineThreads) {
    float o = 0.f;
#pragma unroll 8
    for (int s = 0; s < n; ++s) o = fmaf(coef[s], o0[s * slot_stride + d], o);
    p.out[((size_t)b * p.H_q + j) * Dv + d] = __float2bfloat16_rn(o);
  }
  if (threadIdx.x == 0) p.lse[(size_t)b * p.H_q + j] = lse_out;
}

}  // namespace

cudaError_t launch_combine(const Launch& p, cudaStream_t stream) {
  const long long blocks = (long long)p.B * p.H_q;
  if (blocks == 0) return cudaSuccess;
  return launch_after(combine_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, p);
}

}  // namespace da
