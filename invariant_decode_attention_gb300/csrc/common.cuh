// Shared device helpers and launch descriptors of the decode attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_attn.h"

namespace da {

// ---------------------------------------------------------------------------
// Split constants.  They fix the bits of every output, so they are compile
// time only (never derived from the batch or the GPU).  Per variant:
// tokens per tile, minimum tiles per split, maximum splits per row.
// ---------------------------------------------------------------------------
constexpr int kFmaTile = 64;
constexpr int kFmaMinTilesPerSplit = 16;
constexpr int kFmaMaxSplits = 64;

// CUDA-core variant: query heads per KV head it takes at most.
constexpr int kFmaMaxGroup = 128;

constexpr int kMlaTile = 64;
constexpr int kMlaMinTilesPerSplit = 8;
constexpr int kMlaMaxSplits = 32;

// Tensor-core variant for groups of >= 16 query heads over separate K and V.
constexpr int kTcTile = 64;
constexpr int kTcMinTilesPerSplit = 16;
constexpr int kTcMaxSplits = 64;

// BALANCED quota: tiles charged per split on top of its own tiles, and parts
// the quota divides the batch into per set of CTAs that run one item at once
// (four: every CTA takes several items, so placement can even out the parts).
constexpr int kBalancedFixedOverhead = 2;
constexpr int kBalancedPartsPerSlot = 4;

// Header words at the start of the workspace.
constexpr int kHdrError = 0;  // DA_DEVERR_* bits
constexpr int kHdrNWork = 1;  // number of (row, split) work items
constexpr int kHdrQueue = 2;  // CUDA-core split kernel: units handed out so far
constexpr int kHdrExits = 3;  // CUDA-core split kernel: CTAs that have finished
constexpr int kHdrNEmpty = 4; // work items with no tiles (empty rows); listed last
constexpr size_t kHdrBytes = 256;

// Longest a pipeline wait may spin before the kernel gives up (ns).
constexpr unsigned long long kWaitLimitNs = 4000000000ull;
// The limit of the one wait the time-out test hook (DA_FLAG_TEST_STALL) makes
// run out.
constexpr unsigned long long kTestStallNs = 2000000ull;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Everything a split / combine kernel needs, by value.
struct Launch {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* table;
  const int32_t* lengths;
  __nv_bfloat16* out;
  float* lse;
  int32_t* hdr;
  const int32_t* n_splits;
  const int32_t* split_begin;
  const int32_t* work;
  const int32_t* item_desc;  // int4 per work item: {slot or ~slot if single, tb, te, L}
  float* lse_part;
  float* o_part;
  long long num_blocks;
  // optional second, index-gathered KV source continuing each row's list
  // (extra_k == nullptr: none)
  const __nv_bfloat16* extra_k;
  const __nv_bfloat16* extra_v;
  const int32_t* extra_table;
  const int32_t* extra_lengths;
  long long extra_num_blocks;
  int extra_width;
  int B, H_q, H_kv, D_qk, D_v;
  int layout, page_size, width, capacity;
  int page_shift;  // log2(page_size) when it is a power of two, else -1
  int max_splits;
  float scale_log2;  // softmax scale * log2(e) (* k_scale for an E4M3 cache)
  int kv_type;       // K and V elements: 0 bf16, 1 E4M3 bytes, 2 NVFP4 (codes + block scales)
  long long kv_rows; // NVFP4: rows of the main cache (its block scales follow its codes)
  int o_part_mla;    // partials in the tensor-core variant's head-interleaved layout
  float v_scale;     // E4M3 cache: multiplies each unit's output
  int fma_group;     // CUDA-core variant: query heads per KV head (G)
  int fma_chunks;    // CUDA-core variant: units per KV head (head chunks)
  int test_stall;    // DA_FLAG_TEST_STALL: tensor-core kernels stall at start (tests)
};

struct PlanLaunch {
  const int32_t* lengths;
  const int32_t* extra_lengths;  // nullptr: no second source
  int32_t* hdr;
  int32_t* n_splits;
  int32_t* split_begin;
  int32_t* work;
  int32_t* item_desc;
  int B, tile, min_tps, max_splits, capacity, extra_capacity;
  int policy, num_parts, fixed_overhead;
};

// Launch `kernel` on `stream` so that it may be scheduled while the previous
// kernel on the stream is still running (programmatic dependent launch); the
// kernel calls wait_prior_grid() before reading that kernel's results.
template <typename... Args>
inline cudaError_t launch_after(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Host launchers (each in its own translation unit).
cudaError_t launch_plan(const PlanLaunch& p, cudaStream_t stream);
cudaError_t launch_split_fma(const Launch& p, int grid, cudaStream_t stream);
cudaError_t launch_combine(const Launch& p, cudaStream_t stream);
cudaError_t launch_split_mla(const Launch& p, int grid, cudaStream_t stream);
cudaError_t launch_split_gqa_tc(const Launch& p, int grid, cudaStream_t stream);
bool gqa_tc_supported(int G, int D);
int gqa_tc_resident_ctas(int sms);
// Persistent CTAs that fit on one SM for the variant's split kernel.
int fma_ctas_per_sm(int G, int D);
int mla_resident_ctas(int sms);  // persistent CTAs, an even number
bool fma_supported(int G, int D);
void fma_chunk_shape(int G, int D, int* gc, int* chunks);

// Capacity of a row (largest valid length) for a layout.
inline long long row_capacity(int layout, int width, int page_size) {
  if (layout == DA_KV_PAGED) return (long long)width * page_size;
  return width;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- packed fp32 pairs (one 64-bit register = {lo, hi}) -------------------
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + c on both halves (round to nearest even, no contraction change)
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// bf16 pair (one 32-bit word) -> packed fp32 pair {lo, hi}, exactly.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// bf16 pair (as one 32-bit word) -> two floats, exactly.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete; false if the time limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---- cp.async (16 bytes, L2 only) ------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on the mbarrier at shared address `bar` once every cp.async this
// thread has issued so far has landed.  The arrival is not added to the
// barrier's pending count: its initial count includes it.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Wait until every cp.async this thread has issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 8- and 4-byte copies (through L1; both addresses aligned to the size)
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// ---- low-precision element decoding (all exact) -----------------------------
// Eight E2M1 codes (a 32-bit word, element 2j in the low nibble of byte j) to
// four f16 pairs; pair j holds elements 2j (low half) and 2j + 1.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 codes (low byte first) to an f16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two));
  return h;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// ---- bulk async copy global -> shared (TMA engine, non-tensor form) --------
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- quantized caches on the tensor cores: f16 operands -------------------
// Every E4M3 value is an f16 value, and so is every NVFP4 element (an E2M1
// code, at most two significant bits, times an E4M3 block scale, at most
// four, with magnitudes from 2^-10 to 2688), so K and V convert exactly; Q
// (bf16) is brought into f16's range per row by a power of two: with m the row's
// largest magnitude and 2^k <= m < 2^(k+1), the row is multiplied by
// 2^e, e = 14 - k (clamped to [-113, 120]), so its largest element lies in
// [2^14, 2^15).  Elements below 2^-14 of that (after scaling) become f16
// subnormals, an absolute error of at most 2^-25 * 2^-e, far below the fp32
// accumulation's.  The softmax divides the row's scores by 2^e again.
__device__ __forceinline__ int q_prescale_exp(float maxabs) {
  const uint32_t bits = __float_as_uint(maxabs);
  const int biased = (int)((bits >> 23) & 0xff);
  if (maxabs == 0.f || biased == 0xff) return 0;  // zero row, or inf / NaN: no scaling
  const int k = (biased == 0) ? -127 : biased - 127;
  return min(120, max(-113, 14 - k));
}

// 2^e for e in [-126, 127].
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Largest magnitude of eight bf16 values.
__device__ __forceinline__ float bf16x8_absmax(uint4 w) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(v[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(v[i] & 0xffff0000u)));
  }
  return m;
}

// Running maximum of bf16 magnitudes as integers: the magnitude bits of a
// bf16 (sign cleared) order like the values for every non-NaN value, so
// `acc` keeps, per 16-bit half, the largest magnitude's bits seen so far
// (a NaN's bits sort above infinity's; q_prescale_exp treats both alike).
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint32_t acc, uint4 w) {
  acc = __vmaxu2(acc, w.x & 0x7fff7fffu);
  acc = __vmaxu2(acc, w.y & 0x7fff7fffu);
  acc = __vmaxu2(acc, w.z & 0x7fff7fffu);
  return __vmaxu2(acc, w.w & 0x7fff7fffu);
}

// The fp32 value of the larger of the two magnitudes held by `acc`.
__device__ __forceinline__ float bf16_absmax_value(uint32_t acc) {
  const uint32_t m = max(acc & 0xffffu, acc >> 16);
  return __uint_as_float(m << 16);
}

// Barrier over `n` threads that also returns the OR of `pred` across them.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before the previous kernel on the stream ends; it
// must wait here before touching anything that kernel writes.  Without such
// a predecessor the wait returns at once.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel on the stream (if launched with programmatic stream
// serialisation) be scheduled now; it still waits for this grid to finish.
__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_error(int32_t* hdr, int bits) {
  atomicOr(reinterpret_cast<int*>(hdr + kHdrError), bits);
}

// A row's length after the same clamp the plan applies.
__device__ __forceinline__ int clamp_len(int L, int capacity) {
  return L < 0 ? 0 : (L > capacity ? capacity : L);
}

#endif  // __CUDACC__

}  // namespace da
