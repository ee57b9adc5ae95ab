// Combine kernel: fixed-order fp32 log-sum-exp merge of the split partials of
// every (row b, query head j) whose row has n > 1 splits (the arithmetic is
// in merge.cuh).  The partial LSEs are kept in log2 units by the split
// kernel.  n depends only on the row's own length under the INVARIANT plan,
// so the addends and their order are the same in any batch.
//
// One CTA per (row, head): every thread owns up to four value dims (d,
// d + 128, ...).  It loads its values of a batch of kBatch splits first (all
// those loads in flight at once: a row of 64 splits costs four round trips to
// L2, not 64; the first batch is issued before warp 0 forms the weights),
// then advances its FMA chains through the batch; each chain runs in split
// order from zero, as merge.cuh states.
#include "common.cuh"
#include "merge.cuh"

namespace da {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kMaxDimsPerThread = 4;  // D_v <= 512
constexpr int kBatch = 16;            // splits whose loads are issued together
constexpr int kMaxSplitsAny = kFmaMaxSplits > kMlaMaxSplits ? kFmaMaxSplits : kMlaMaxSplits;
static_assert(kMaxSplitsAny <= 64, "two split weights per lane of warp 0");

// DPT: value dims per thread (1 when D_v <= 128, else up to 4).
template <int DPT>
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
  float v[kBatch][DPT];
  auto load = [&](int s0) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
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
  for (int s0 = 0; s0 < n; s0 += kBatch) {
    if (s0 > 0) load(s0);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
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

// The tensor-core variant's partials are head-interleaved: value dims in
// groups of four, heads innermost -- element (slot, head j, dim d) at
// ((slot * 128 + d / 4) * H_q + j) * 4 + d % 4 -- so that its epilogue's
// stores coalesce.  Its combine takes one CTA per (row, value half, 32 dims)
// and one thread per head: each thread forms its head's weights alone with
// the same operations in the same order as merge_weights (its weights sit in
// a shared-memory column; the split LSEs are loaded together), and its loads
// of a split's 4-dim group coalesce across the heads.  The loads of two
// splits are issued before their FMAs, the first two before the weights are
// formed.
constexpr int kMlaGroupsPerCta = 8;  // 4-dim groups: 32 value dims
constexpr int kMlaBatch = 2;         // splits whose loads are issued together

__global__ void __launch_bounds__(kCombineThreads) combine_mla_kernel(Launch p) {
  wait_prior_grid();  // the split kernel's partials
  constexpr int kBlocksPerRow = 512 / 4 / kMlaGroupsPerCta;  // 16
  const int b = blockIdx.x / kBlocksPerRow, cb = blockIdx.x % kBlocksPerRow;
  const int n = p.n_splits[b];
  const int j = threadIdx.x;
  if (n <= 1 || j >= p.H_q) return;
  const size_t slot0 = (size_t)b * p.max_splits;
  __shared__ float coef_s[kMlaMaxSplits][kCombineThreads];
  const float4* base = reinterpret_cast<const float4*>(p.o_part) +
                       (slot0 * 128 + cb * kMlaGroupsPerCta) * p.H_q + j;
  float4 v[kMlaBatch][kMlaGroupsPerCta];
  auto load = [&](int s0) {
#pragma unroll
    for (int i = 0; i < kMlaBatch; ++i) {
      const float4* src = base + (size_t)(s0 + i) * 128 * p.H_q;
#pragma unroll
      for (int gi = 0; gi < kMlaGroupsPerCta; ++gi)
        v[i][gi] = (s0 + i < n) ? __ldcg(src + gi * p.H_q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load(0);  // in flight while the weights are formed
  // the split LSEs, all loads issued together
  float ls[kMlaMaxSplits];
#pragma unroll
  for (int s = 0; s < kMlaMaxSplits; ++s)
    ls[s] = (s < n) ? __ldcg(p.lse_part + (slot0 + s) * p.H_q + j) : -INFINITY;
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMlaMaxSplits; ++s) M = fmaxf(M, ls[s]);
  float W = 0.f;
#pragma unroll
  for (int s = 0; s < kMlaMaxSplits; ++s) {
    if (s < n) {
      coef_s[s][j] = (M == -INFINITY) ? 0.f : ex2(ls[s] - M);
      W += coef_s[s][j];
    }
  }
  for (int s = 0; s < n; ++s) coef_s[s][j] = (W > 0.f) ? coef_s[s][j] / W : 0.f;
  float4 acc[kMlaGroupsPerCta];
#pragma unroll
  for (int gi = 0; gi < kMlaGroupsPerCta; ++gi) acc[gi] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += kMlaBatch) {
    if (s0 > 0) load(s0);
#pragma unroll
    for (int i = 0; i < kMlaBatch; ++i) {
      if (s0 + i < n) {
        const float c = coef_s[s0 + i][j];
#pragma unroll
        for (int gi = 0; gi < kMlaGroupsPerCta; ++gi) {
          acc[gi].x = fmaf(c, v[i][gi].x, acc[gi].x);
          acc[gi].y = fmaf(c, v[i][gi].y, acc[gi].y);
          acc[gi].z = fmaf(c, v[i][gi].z, acc[gi].z);
          acc[gi].w = fmaf(c, v[i][gi].w, acc[gi].w);
        }
      }
    }
  }
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(
      p.out + ((size_t)b * p.H_q + j) * 512 + cb * kMlaGroupsPerCta * 4);
#pragma unroll
  for (int gi = 0; gi < kMlaGroupsPerCta; ++gi) {
    dst[2 * gi] = __floats2bfloat162_rn(acc[gi].x, acc[gi].y);
    dst[2 * gi + 1] = __floats2bfloat162_rn(acc[gi].z, acc[gi].w);
  }
  if (cb == 0) p.lse[(size_t)b * p.H_q + j] = (W > 0.f) ? (M + lg2(W)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Launch& p, cudaStream_t stream) {
  if (p.o_part_mla) {
    if (p.D_v != 512 || p.H_q > kCombineThreads) return cudaErrorInvalidValue;
    const long long blocks = (long long)p.B * (512 / 4 / kMlaGroupsPerCta);
    if (blocks == 0) return cudaSuccess;
    return launch_after(combine_mla_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0,
                        stream, p);
  }
  if (p.D_v > kCombineThreads * kMaxDimsPerThread) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.B * p.H_q;
  if (blocks == 0) return cudaSuccess;
  if (p.D_v <= kCombineThreads)
    return launch_after(combine_kernel<1>, dim3((unsigned)blocks), dim3(kCombineThreads), 0,
                        stream, p);
  return launch_after(combine_kernel<kMaxDimsPerThread>, dim3((unsigned)blocks),
                      dim3(kCombineThreads), 0, stream, p);
}

}  // namespace da
