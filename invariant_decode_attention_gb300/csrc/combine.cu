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
#include "common.cuh"

namespace da {
namespace {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(Launch p) {
  __shared__ float coef[kCombineWarps][kFmaMaxSplits > kMlaMaxSplits ? kFmaMaxSplits : kMlaMaxSplits];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kCombineWarps + warp;
  if (gw >= (long long)p.B * p.H_q) return;
  const int b = (int)(gw / p.H_q), j = (int)(gw % p.H_q);
  const int n = p.n_splits[b];
  if (n <= 1) return;  // written final by the split kernel
  const size_t slot0 = (size_t)b * p.max_splits;
  float lse_s[2];
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = lane + 32 * i;
    lse_s[i] = (s < n) ? p.lse_part[(slot0 + s) * p.H_q + j] : -INFINITY;
    M = fmaxf(M, lse_s[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float* cw = coef[warp];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = lane + 32 * i;
    if (s < n) cw[s] = (M == -INFINITY) ? 0.f : ex2(lse_s[i] - M);
  }
  __syncwarp();
  float W = 0.f;
  for (int s = 0; s < n; ++s) W += cw[s];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = lane + 32 * i;
    if (s < n) cw[s] = (W > 0.f) ? cw[s] / W : 0.f;
  }
  __syncwarp();
  const int Dv = p.D_v;
  const float* o0 = p.o_part + (slot0 * p.H_q + j) * (size_t)Dv;
  const size_t slot_stride = (size_t)p.H_q * Dv;
  for (int d = lane; d < Dv; d += 32) {
    float o = 0.f;
    for (int s = 0; s < n; ++s) o = fmaf(cw[s], o0[s * slot_stride + d], o);
    p.out[((size_t)b * p.H_q + j) * Dv + d] = __float2bfloat16_rn(o);
  }
  if (lane == 0) p.lse[(size_t)b * p.H_q + j] = (W > 0.f) ? (M + lg2(W)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Launch& p, cudaStream_t stream) {
  const long long warps = (long long)p.B * p.H_q;
  if (warps == 0) return cudaSuccess;
  const long long blocks = (warps + kCombineWarps - 1) / kCombineWarps;
  combine_kernel<<<(unsigned)blocks, kCombineWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace da
