// Fixed-order fp32 log-sum-exp merge of one (row, query head)'s split
// results: the combine step of "Sparse MLA decode is not batch-invariant"
// (FlashMLA issue #212, section "Where it comes from": every split's output
// rescaled by its LSE and summed in split order), with the split count taken
// from the per-row plan.  For n partials with LSEs lse_s (log2 units) and
// outputs o_s:
//     M   = max_s lse_s
//     w_s = 2^(lse_s - M),   W = w_0 + w_1 + ... + w_{n-1}   (in this order)
//     out = sum_s (w_s / W) * o_s                            (fp32, s ascending)
//     lse = (M + log2 W) * ln 2                              (natural log)
// merge_weights forms the weights; the value sums are fp32 FMA chains
// acc = fma(w_s / W, o_s, acc) from acc = 0, s ascending.
#pragma once

#include "common.cuh"

namespace da {

// Weights coef[0..n) (n <= 64) of a (row, head)'s partials whose LSEs sit at
// lse[s * stride]; coef is shared memory.  Called by one whole warp; returns
// the merged LSE (natural log) in every lane.  Partials written by other
// CTAs of the running kernel are read through L2 (ld.global.cg).
__device__ __forceinline__ float merge_weights(const float* lse, size_t stride, int n,
                                               float* coef, int lane) {
  float ls[2];
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = lane + 32 * i;
    ls[i] = (s < n) ? __ldcg(lse + (size_t)s * stride) : -INFINITY;
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
  __syncwarp();
  return (W > 0.f) ? (M + lg2(W)) * kLn2 : -INFINITY;
}

// The combine launch for partials whose rows have at most n_bound splits
// each (a bound the plan implies: its kernel then keeps no registers for
// splits beyond it).
cudaError_t launch_combine(const Launch& p, int n_bound, cudaStream_t stream);

}  // namespace da
