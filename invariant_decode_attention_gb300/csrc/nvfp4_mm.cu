// Batch-invariant NVFP4 weight matmul y = global_scale * bf16(x) @ W^T.
//
// "Greedy outputs depend on batch composition" (gllm issue #98, Candidate
// cause) finds a weight matmul whose kernel -- and with it the activation
// precision -- is picked by the row count n; its Next steps propose one
// activation precision, bf16, for every n.  Here every n also gets one
// arithmetic: the tensor core computes every tile the same way, K is cut into
// fixed chunks of NVFP4_MM_K_CHUNK whatever n is, and the chunk sums are
// added in chunk order.  A row's bits therefore depend on its own activations
// and the weight only.
//
// Tile: 128 output features (MMA M, one per tensor-memory lane) x 32
// activation rows (MMA N) x one K chunk; the MMA is D[o, i] += W[o, k] x[i, k]
// ("swap AB": the weight is the 128-row operand, so a small n wastes nothing
// of the weight stream).  Per 64-wide K step of the chunk:
//   warp 0     TMA: the step's 128 x 32 bytes of E2M1 codes into a 6-deep
//              ring (no swizzle), the step's 32 x 64 bf16 activations into a
//              4-deep ring (128-byte swizzle, K-major);
//   warps 2-5  dequantize: thread r owns weight row r of the tile, decodes
//              its 64 codes with the row's four E4M3 block scales into bf16
//              (exact: an E2M1 value times an E4M3 scale has at most six
//              significant bits) and writes them into a 3-deep ring in the
//              128-byte-swizzled K-major layout the tensor core reads;
//   warp 1     MMA issue (one thread): four M128 N32 K16 MMAs into a 32-column
//              fp32 accumulator in tensor memory.
// After the chunk, warps 2-5 read the accumulator (thread r = lane r) and
// write the chunk's partial sums, or y itself when K is a single chunk.
// Every mbarrier wait is bounded; on time-out the kernel records
// DA_DEVERR_TIMEOUT, all roles leave their loops, the copies in flight and
// the tensor-core work are drained (bounded) and tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "nvfp4_mm.h"
#include "tcgen05.cuh"

namespace da {
namespace {

constexpr int kTileN = NVFP4_MM_TILE_N;     // weight rows per tile (MMA M)
constexpr int kRowTile = NVFP4_MM_ROW_TILE; // activation rows per tile (MMA N)
constexpr int kKChunk = NVFP4_MM_K_CHUNK;   // K per partial sum
constexpr int kStep = 64;                   // K per pipeline step (one swizzle row)
constexpr int kStepsPerChunk = kKChunk / kStep;
constexpr int kRawStages = 6, kXStages = 4, kAStages = 3;
constexpr int kRawBytes = kTileN * kStep / 2;   // 4096: E2M1 codes of a step
constexpr int kXBytes = kRowTile * kStep * 2;   // 4096: bf16 activations of a step
constexpr int kABytes = kTileN * kStep * 2;     // 16384: bf16 weights of a step
constexpr int kScaleStride = kStepsPerChunk * 4 + 4;  // 68 bytes per row: no bank conflicts

constexpr int kAOff = 0;
constexpr int kXOff = kAOff + kAStages * kABytes;        // 49152
constexpr int kRawOff = kXOff + kXStages * kXBytes;      // 65536
constexpr int kScaleOff = kRawOff + kRawStages * kRawBytes;  // 90112
constexpr int kBarOff = kScaleOff + kTileN * kScaleStride;   // 98816
enum { kRawFull0 = 0, kRawEmpty0 = kRawFull0 + kRawStages, kXFull0 = kRawEmpty0 + kRawStages,
       kXEmpty0 = kXFull0 + kXStages, kAFull0 = kXEmpty0 + kXStages,
       kAEmpty0 = kAFull0 + kAStages, kDFull = kAEmpty0 + kAStages, kDrain, kNumBars };
constexpr int kTmemSlot = kBarOff + kNumBars * 8;
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kSmemBytes = kAbortSlot + 4;
static_assert(kXOff % 1024 == 0 && kABytes % 1024 == 0 && kXBytes % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(kBarOff % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kIdesc = umma::idesc_bf16_f32(kTileN, kRowTile, false);

struct MmArgs {
  const uint8_t* scales;  // [N, K / 16]
  float* part;            // [n_chunks, n, N] partial sums (n_chunks > 1)
  float* y;               // [n, N]
  __nv_bfloat16* y_bf16;  // [n, N] or null
  int32_t* hdr;           // workspace header (error word)
  float global_scale;
  int n, N, K, n_chunks, n_itiles;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Eight E2M1 codes (a 32-bit word, code 2j in the low nibble of byte j) to
// four f16 pairs, code 2j in the low half of pair j (exact).
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

// Two E4M3 codes (low byte first) to an f16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two));
  return h;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// An f16 pair holding values exactly representable in bf16 -> bf16 pair.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  volatile int* abort_flag;
  int32_t* hdr;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) {
  return c.sbase + kBarOff + 8 * i;
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_bar(const Ctx& c, int i, uint32_t parity) {
  const uint32_t bar = bar_addr(c, i);
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*c.abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_error(c.hdr, DA_DEVERR_TIMEOUT);
        *c.abort_flag = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- roles

__device__ void producer(const Ctx& c, const CUtensorMap* tm_w, const CUtensorMap* tm_x,
                         int o0, int i0, int k0, int n_steps) {
  int w_issued = 0, x_issued = 0;
  auto issue_w = [&](int j) -> bool {
    const int s = j % kRawStages;
    if (j >= kRawStages && !wait_bar(c, kRawEmpty0 + s, ((j / kRawStages) - 1) & 1)) return false;
    mbar_arrive_expect_tx(bar_addr(c, kRawFull0 + s), kRawBytes);
    tma_load_2d(c.sbase + kRawOff + s * kRawBytes, tm_w, (k0 + j * kStep) / 2, o0,
                bar_addr(c, kRawFull0 + s));
    w_issued = j + 1;
    return true;
  };
  // The weight does not come from the previous kernel on the stream: start
  // streaming it before waiting for that kernel (which writes the activations).
  bool ok = true;
  for (int j = 0; j < n_steps && j < kRawStages && ok; ++j) ok = issue_w(j);
  wait_prior_grid();
  for (int j = 0; j < n_steps && ok; ++j) {
    const int s = j % kXStages;
    if (j >= kXStages && !wait_bar(c, kXEmpty0 + s, ((j / kXStages) - 1) & 1)) break;
    mbar_arrive_expect_tx(bar_addr(c, kXFull0 + s), kXBytes);
    tma_load_2d(c.sbase + kXOff + s * kXBytes, tm_x, k0 + j * kStep, i0, bar_addr(c, kXFull0 + s));
    x_issued = j + 1;
    if (j + kRawStages < n_steps) ok = issue_w(j + kRawStages);
  }
  // Copies still in flight must land before the CTA's shared memory goes away.
  for (int s = 0; s < kRawStages; ++s) {
    const int last = w_issued - 1 - ((w_issued - 1 - s) % kRawStages + kRawStages) % kRawStages;
    if (last >= 0 && !mbar_wait(bar_addr(c, kRawFull0 + s), (last / kRawStages) & 1))
      set_error(c.hdr, DA_DEVERR_TIMEOUT);
  }
  for (int s = 0; s < kXStages; ++s) {
    const int last = x_issued - 1 - ((x_issued - 1 - s) % kXStages + kXStages) % kXStages;
    if (last >= 0 && !mbar_wait(bar_addr(c, kXFull0 + s), (last / kXStages) & 1))
      set_error(c.hdr, DA_DEVERR_TIMEOUT);
  }
}

__device__ void mma_issuer(const Ctx& c, uint32_t tmem, int n_steps) {
  for (int j = 0; j < n_steps; ++j) {
    const int sa = j % kAStages, sx = j % kXStages;
    if (!wait_bar(c, kAFull0 + sa, (j / kAStages) & 1)) return;
    if (!wait_bar(c, kXFull0 + sx, (j / kXStages) & 1)) return;
    umma::fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < kStep / 16; ++kk) {  // K = 16 per MMA: 32 bytes along the row
      const uint64_t a = umma::smem_desc(c.sbase + kAOff + sa * kABytes + kk * 32, 16, 1024,
                                         umma::kSwizzle128B);
      const uint64_t b = umma::smem_desc(c.sbase + kXOff + sx * kXBytes + kk * 32, 16, 1024,
                                         umma::kSwizzle128B);
      umma::mma_bf16(tmem, a, b, kIdesc, (j | kk) ? 1u : 0u);
    }
    umma::commit(bar_addr(c, kAEmpty0 + sa));
    umma::commit(bar_addr(c, kXEmpty0 + sx));
  }
  umma::commit(bar_addr(c, kDFull));
}

// Thread r (0..127) of warps 2-5: weight row r of the tile, which is also
// tensor-memory lane r for the epilogue (a warp reads lanes 32 (warp % 4)..).
__device__ void dequant_and_store(const Ctx& c, const MmArgs& a, uint32_t tmem, int o0, int i0,
                                  int chunk, int k0, int n_steps) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;
  const bool leader = lane == 0;
  // the chunk's block scales of row r: n_steps words of four E4M3 codes
  {
    const uint8_t* src = a.scales + (size_t)(o0 + r) * (a.K / 16) + k0 / 16;
    const uint32_t dst = c.sbase + kScaleOff + r * kScaleStride;
    for (int j = 0; j < n_steps; ++j) cp_async4(dst + 4 * j, src + 4 * j);
    cp_async_commit();
  }
  const uint8_t* srow = c.smem + kScaleOff + r * kScaleStride;
  cp_async_wait<0>();
  bool ok = true;
  for (int j = 0; j < n_steps && ok; ++j) {
    const int s = j % kRawStages, sa = j % kAStages;
    if (!wait_bar(c, kRawFull0 + s, (j / kRawStages) & 1)) { ok = false; break; }
    const uint8_t* raw = c.smem + kRawOff + s * kRawBytes + r * (kStep / 2);
    const uint4 w0 = *reinterpret_cast<const uint4*>(raw);
    const uint4 w1 = *reinterpret_cast<const uint4*>(raw + 16);
    __syncwarp();
    if (leader) mbar_arrive(bar_addr(c, kRawEmpty0 + s));
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(srow + 4 * j);
    const uint32_t s01 = e4m3x2_to_f16x2(sw & 0xffffu), s23 = e4m3x2_to_f16x2(sw >> 16);
    const uint32_t sc[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                            __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    if (j >= kAStages && !wait_bar(c, kAEmpty0 + sa, ((j / kAStages) - 1) & 1)) { ok = false; break; }
    uint8_t* arow = c.smem + kAOff + sa * kABytes + r * 128;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {  // 16-byte chunk cc: weights 8cc .. 8cc+7
      uint32_t h[4], o[4];
      e2m1x8_to_f16x2(words[cc], h);
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = f16x2_to_bf16x2(hmul2(h[q], sc[cc >> 1]));
      *reinterpret_cast<uint4*>(arow + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async();
    __syncwarp();
    if (leader) mbar_arrive(bar_addr(c, kAFull0 + sa));
  }
  if (!ok || !wait_bar(c, kDFull, 0)) return;
  umma::fence_after_sync();
  float v[32];
  umma::ld_32x32b_x32(tmem + ((uint32_t)((warp & 3) * 32) << 16), v);
  umma::wait_ld();
  const int o = o0 + r;
  const int rows = min(kRowTile, a.n - i0);
  if (a.n_chunks == 1) {
#pragma unroll
    for (int q = 0; q < kRowTile; ++q) {
      if (q < rows) {
        const float yv = a.global_scale * v[q];
        a.y[(size_t)(i0 + q) * a.N + o] = yv;
        if (a.y_bf16) a.y_bf16[(size_t)(i0 + q) * a.N + o] = __float2bfloat16_rn(yv);
      }
    }
  } else {
    float* dst = a.part + ((size_t)chunk * a.n + i0) * a.N + o;
#pragma unroll
    for (int q = 0; q < kRowTile; ++q)
      if (q < rows) dst[(size_t)q * a.N] = v[q];
  }
}

// Tile id -> (activation tile, chunk, weight tile); activation tiles of one
// weight chunk are neighbours, so they run together and share it in L2.
__global__ void __launch_bounds__(kThreads, 2)
    nvfp4_mm_kernel(MmArgs a, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_x) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
  c.hdr = a.hdr;
  const int warp = threadIdx.x >> 5;
  allow_next_grid();  // the combine kernel may be scheduled; it waits for this grid
  const int id = blockIdx.x;
  const int it = id % a.n_itiles;
  const int rest = id / a.n_itiles;
  const int chunk = rest % a.n_chunks;
  const int o0 = (rest / a.n_chunks) * kTileN, i0 = it * kRowTile;
  const int k0 = chunk * kKChunk;
  const int n_steps = (min(a.K, k0 + kKChunk) - k0) / kStep;
  if (c.sbase & 1023u) {  // the swizzled layouts need 1024-byte-aligned shared memory
    if (threadIdx.x == 0) set_error(a.hdr, DA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;  // TMA expect_tx arrive or tcgen05.commit
      if ((i >= kRawEmpty0 && i < kRawEmpty0 + kRawStages) ||
          (i >= kAFull0 && i < kAFull0 + kAStages))
        count = 4;         // one arrive per dequantizing warp
      mbar_init(bar_addr(c, i), count);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    umma::tmem_alloc(c.sbase + kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) producer(c, &tm_w, &tm_x, o0, i0, k0, n_steps);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) {
      mma_issuer(c, tmem, n_steps);
      umma::commit(bar_addr(c, kDrain));  // arrives once every MMA above has completed
    }
  } else {
    // Its stores come after the MMAs, which come after the producer's wait
    // for the previous kernel: they never overtake that kernel's reads.
    dequant_and_store(c, a, tmem, o0, i0, chunk, k0, n_steps);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    umma::fence_after_sync();
    if ((threadIdx.x & 31) == 0 && !mbar_wait(bar_addr(c, kDrain), 0))
      set_error(a.hdr, DA_DEVERR_TIMEOUT);
    __syncwarp();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// fp32 / bf16 activations [n, K] -> bf16 [n_pad, K] (round to nearest even),
// rows n .. n_pad - 1 zero.  Eight elements per thread and step.
__global__ void nvfp4_round_kernel(const void* x, int x_dtype, __nv_bfloat16* xr, int32_t* hdr,
                                   int n, int n_pad, int K) {
  wait_prior_grid();
  allow_next_grid();  // after the wait: the next kernel may read the weight early
  if (blockIdx.x == 0 && threadIdx.x == 0) hdr[kHdrError] = 0;  // errors of this call only
  const size_t total = (size_t)n_pad * K / 8, valid = (size_t)n * K / 8;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < total;
       v += (size_t)gridDim.x * blockDim.x) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (v < valid) {
      if (x_dtype == NVFP4_X_F32) {
        const float4 f0 = __ldg(reinterpret_cast<const float4*>(x) + 2 * v);
        const float4 f1 = __ldg(reinterpret_cast<const float4*>(x) + 2 * v + 1);
        __nv_bfloat162 b0 = __floats2bfloat162_rn(f0.x, f0.y), b1 = __floats2bfloat162_rn(f0.z, f0.w);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f1.x, f1.y), b3 = __floats2bfloat162_rn(f1.z, f1.w);
        o = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                       *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
      } else {
        o = __ldg(reinterpret_cast<const uint4*>(x) + v);
      }
    }
    reinterpret_cast<uint4*>(xr)[v] = o;
  }
}

// y = global_scale * (((P_0 + P_1) + P_2) + ...), four outputs per thread.
__global__ void nvfp4_combine_kernel(const float* part, float* y, __nv_bfloat16* y_bf16,
                                     float global_scale, int n_chunks, size_t count) {
  wait_prior_grid();
  const size_t n4 = count / 4;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n4;
       v += (size_t)gridDim.x * blockDim.x) {
    float4 s = __ldg(reinterpret_cast<const float4*>(part) + v);
    for (int ch = 1; ch < n_chunks; ++ch) {
      const float4 p = __ldg(reinterpret_cast<const float4*>(part + (size_t)ch * count) + v);
      s.x += p.x;
      s.y += p.y;
      s.z += p.z;
      s.w += p.w;
    }
    s.x *= global_scale;
    s.y *= global_scale;
    s.z *= global_scale;
    s.w *= global_scale;
    reinterpret_cast<float4*>(y)[v] = s;
    if (y_bf16) {
      __nv_bfloat162 b0 = __floats2bfloat162_rn(s.x, s.y), b1 = __floats2bfloat162_rn(s.z, s.w);
      reinterpret_cast<uint2*>(y_bf16)[v] =
          make_uint2(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1));
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

constexpr size_t kHdr = 256;

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

int n_chunks_of(int K) { return (K + kKChunk - 1) / kKChunk; }

size_t xr_bytes(int n, int K) { return round_up((size_t)round_up(n, kRowTile) * K * 2, 256); }

bool shape_ok(int n, int N, int K) {
  if (n < 0 || N <= 0 || K <= 0 || N % kTileN || K % kStep) return false;
  if ((long long)round_up(n, kRowTile) * K >= (1ll << 31) || (long long)n * N >= (1ll << 31))
    return false;
  return true;
}

}  // namespace
}  // namespace da

using namespace da;

extern "C" {

size_t nvfp4_mm_workspace_bytes(int32_t n, int32_t N, int32_t K) {
  if (!shape_ok(n, N, K)) return 0;
  const int nc = n_chunks_of(K);
  size_t b = kHdr + xr_bytes(n, K);
  if (nc > 1) b += round_up((size_t)nc * n * N * 4, 256);
  return b;
}

int nvfp4_mm(const void* x, int32_t x_dtype, const uint8_t* codes, const uint8_t* scales,
             float global_scale, int32_t n, int32_t N, int32_t K, float* y, void* y_bf16,
             void* ws, size_t ws_bytes, void* stream) {
  if (x_dtype != NVFP4_X_F32 && x_dtype != NVFP4_X_BF16) return DA_ERR_INVALID_ARG;
  if (!(global_scale == global_scale) || global_scale - global_scale != 0.f)
    return DA_ERR_INVALID_ARG;  // NaN or infinite
  if (!shape_ok(n, N, K)) return DA_ERR_UNSUPPORTED;
  if (n == 0) return DA_OK;
  if (!x || !codes || !scales || !y) return DA_ERR_INVALID_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)codes & 15) || ((uintptr_t)scales & 3) ||
      ((uintptr_t)y & 15) || ((uintptr_t)y_bf16 & 7))
    return DA_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & 255)) return DA_ERR_WORKSPACE;
  if (ws_bytes < nvfp4_mm_workspace_bytes(n, N, K)) return DA_ERR_WORKSPACE;
  const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return DA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int n_pad = (int)round_up(n, kRowTile);
  const int nc = n_chunks_of(K);
  uint8_t* base = static_cast<uint8_t*>(ws);
  __nv_bfloat16* xr = reinterpret_cast<__nv_bfloat16*>(base + kHdr);
  float* part = nc > 1 ? reinterpret_cast<float*>(base + kHdr + xr_bytes(n, K)) : nullptr;

  alignas(64) CUtensorMap tm_w, tm_x;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {kStep / 2, kTileN};
    const cuuint32_t elem[2] = {1, 1};
    if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
            box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DA_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)n_pad};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {kStep, kRowTile};
    const cuuint32_t elem[2] = {1, 1};
    if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xr, dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DA_ERR_CUDA;
  }
  static const cudaError_t attr = cudaFuncSetAttribute(
      nvfp4_mm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (attr != cudaSuccess) return DA_ERR_CUDA;

  MmArgs a;
  a.scales = scales;
  a.part = part;
  a.y = y;
  a.y_bf16 = static_cast<__nv_bfloat16*>(y_bf16);
  a.hdr = static_cast<int32_t*>(ws);
  a.global_scale = global_scale;
  a.n = n;
  a.N = N;
  a.K = K;
  a.n_chunks = nc;
  a.n_itiles = n_pad / kRowTile;

  const size_t vec = (size_t)n_pad * K / 8;
  const int round_blocks = (int)std::min<size_t>((vec + 255) / 256, 4096);
  if (launch_after(nvfp4_round_kernel, dim3(round_blocks), dim3(256), 0, st, x, (int)x_dtype, xr,
                   a.hdr, (int)n, n_pad, (int)K) != cudaSuccess)
    return DA_ERR_CUDA;
  const long long tiles = (long long)(N / kTileN) * nc * a.n_itiles;
  if (tiles >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
  if (launch_after(nvfp4_mm_kernel, dim3((unsigned)tiles), dim3(kThreads), (size_t)kSmemBytes, st,
                   a, tm_w, tm_x) != cudaSuccess)
    return DA_ERR_CUDA;
  if (nc > 1) {
    const size_t count = (size_t)n * N;
    const int blocks = (int)std::min<size_t>((count / 4 + 255) / 256, 4096);
    if (launch_after(nvfp4_combine_kernel, dim3(blocks), dim3(256), 0, st, (const float*)part, y,
                     a.y_bf16, global_scale, nc, count) != cudaSuccess)
      return DA_ERR_CUDA;
  }
  return DA_OK;
}

int nvfp4_mm_read_error(void* ws, int32_t* code, void* stream) {
  if (!ws || !code) return DA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DA_ERR_CUDA;
  *code = v;
  if (v && cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

}  // extern "C"
