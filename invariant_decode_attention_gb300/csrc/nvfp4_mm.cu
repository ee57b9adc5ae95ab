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
// Work unit ("tile"): 128 output features (MMA M, one per tensor-memory lane)
// x 32 activation rows (MMA N) x one K chunk; the MMA is D[o, i] += W[o, k]
// x[i, k] ("swap AB": the weight is the 128-row operand, so a small n wastes
// nothing of the weight stream).  The kernel is persistent, one CTA per SM,
// each CTA taking tiles blockIdx.x, + gridDim.x, ...; its rings run on across
// tiles, so the next tile's copies and dequantization overlap the current
// tile's MMAs and epilogue.  Per 256-wide K step:
//   16 warps    dequantize: thread (r, b) owns weight row r of the tile and two
//               16-weight blocks of each 128-wide half of the step; it fetches
//               its own 2 x 16 bytes of codes and 2 words of block scales with
//               cp.async two steps ahead (a ring only it reads), decodes them
//               exactly to bf16 (an E2M1 value times an E4M3 scale has at most
//               six significant bits) and writes them into a 2-deep ring in
//               the 128-byte-swizzled K-major layout the tensor core reads;
//   warp 5      TMA (one thread): the step's 32 x 256 bf16 activations into a
//               2-deep ring (128-byte swizzle, K-major);
//   warp 1      MMA issue (one thread): sixteen M128 N32 K16 MMAs per step into
//               one of two 32-column fp32 accumulators in tensor memory (tiles
//               alternate between them); a step's weights and activations
//               complete one barrier, and one commit frees both slots;
//   warps 21-24 epilogue: read a finished accumulator (warp w reads lanes
//               32 (w % 4)..), free it, and write y when K is one chunk, else
//               the chunk's partial sums; the last of a tile's chunk CTAs to
//               finish (a counter per output tile) adds the partials in chunk
//               order and writes y.
// Warp w issues on scheduler w % 4: the pacing single-thread roles (MMA issue,
// activation copies) have scheduler 1 to themselves, the dequantizing warps
// fill the other three.
// One CTA per SM: two CTAs of an earlier version of this kernel sharing an SM
// were measured to corrupt the accumulators of one of them now and then
// (cause not found), so the shared-memory request keeps a second one out.
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
constexpr int kStep = 256;                  // K per pipeline step: four 64-wide swizzle regions
constexpr int kSub = 128;                   // K a dequantizing thread covers per half step: 32
constexpr int kRegion = 64;                 // K of one 128-byte swizzle row of bf16
constexpr int kRegions = kStep / kRegion;
constexpr int kRawStages = 3;               // per-thread code ring (cp.async)
constexpr int kAStages = 2, kXStages = 2;   // weight and activation operand rings
static_assert(kXStages % kAStages == 0, "a step's barriers index both rings");
constexpr int kRawBytes = kTileN * kStep / 2;       // 16384: E2M1 codes of a step
constexpr int kSBytes = 512 * 8;                    // 4096: two 4-byte scale words per dequantizing thread
constexpr int kXRegionBytes = kRowTile * kRegion * 2;  // 4096
constexpr int kXBytes = kRegions * kXRegionBytes;   // 16384: bf16 activations of a step
constexpr int kARegionBytes = kTileN * kRegion * 2;  // 16384
constexpr int kABytes = kRegions * kARegionBytes;   // 65536: bf16 weights of a step

constexpr int kAOff = 0;
constexpr int kXOff = kAOff + kAStages * kABytes;            // 131072
constexpr int kRawOff = kXOff + kXStages * kXBytes;          // 163840
constexpr int kSOff = kRawOff + kRawStages * kRawBytes;      // 212992
constexpr int kBarOff = kSOff + kRawStages * kSBytes;        // 225280
// Step g: its activations (slot g % kXStages) and its weights (slot
// g % kAStages) complete full[g % kXStages]; one commit to empty[g % kXStages]
// frees both slots.
enum { kFull0 = 0, kEmpty0 = kFull0 + kXStages, kDFull0 = kEmpty0 + kXStages,
       kDEmpty0 = kDFull0 + 2, kDrain = kDEmpty0 + 2, kNumBars };
constexpr int kTmemSlot = kBarOff + kNumBars * 8;
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kLastSlot = kAbortSlot + 4;
constexpr int kSmemBytes = kLastSlot + 4;
static_assert(kXOff % 1024 == 0 && kARegionBytes % 1024 == 0 && kXRegionBytes % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(kBarOff % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(kSmemBytes <= 232448 && 2 * (kSmemBytes + 1024) > 233472,
              "fits one CTA per SM and keeps a second one out");

// Warp w issues on scheduler w % 4.  The single-thread roles that set the
// pace (MMA issue, activation copies) get scheduler 1 to themselves; the 16
// dequantizing warps fill schedulers 0, 2 and 3 (ids 0..20 with w % 4 != 1);
// the epilogue needs one warp per tensor-memory lane quarter (w % 4 = 0..3).
constexpr int kMmaWarp = 1, kXWarp = 5;
constexpr int kDqWarps = 16, kDqLastWarp = 20;
constexpr int kEpWarp0 = 21, kEpWarps = 4;   // warps 21..24
static_assert(kRawBytes == kDqWarps * 32 * 32 && kSBytes == kDqWarps * 32 * 8,
              "per-thread code and scale slots fill their stages exactly");
constexpr int kEpThreads = kEpWarps * 32;
constexpr int kThreads = (kEpWarp0 + kEpWarps) * 32;  // 800 (warps 9, 13, 17 idle)
__host__ __device__ constexpr bool is_dq_warp(int w) { return w <= kDqLastWarp && (w & 3) != 1; }
// index 0..15 of a dequantizing warp: its id less the scheduler-1 ids below it
__host__ __device__ constexpr int dq_index(int w) { return w - (w + 3) / 4; }
static_assert(dq_index(0) == 0 && dq_index(2) == 1 && dq_index(kDqLastWarp) == kDqWarps - 1,
              "dequantizing warps are numbered 0..15");
constexpr int kEpBarrier = 2;                          // named barrier of the epilogue warps
constexpr uint32_t kTmemCols = 2 * kRowTile;           // two accumulators
constexpr uint32_t kIdesc = umma::idesc_bf16_f32(kTileN, kRowTile, false);

struct MmArgs {
  const uint8_t* codes;   // [N, K / 2]
  const uint8_t* scales;  // [N, K / 16]
  float* part;            // [n_chunks, n, N] partial sums (n_chunks > 1)
  float* y;               // [n, N]
  __nv_bfloat16* y_bf16;  // [n, N] or null
  int32_t* hdr;           // workspace header (error word)
  int32_t* tile_count;    // [N / 128, n_itiles] chunk CTAs finished per tile (n_chunks > 1)
  float global_scale;
  int n, N, K, n_chunks, n_itiles, n_tiles;
};

// Tile t -> (activation tile, chunk, weight tile); activation tiles of one
// weight chunk are neighbours, so they run together and share it in L2.
struct Tile {
  int o0, i0, k0, k_len, chunk, n_steps, out_tile;  // k_len: K of the chunk (64 .. 1024)
};

__device__ __forceinline__ Tile tile_of(const MmArgs& a, int t) {
  Tile x;
  const int it = t % a.n_itiles;
  const int rest = t / a.n_itiles;
  x.chunk = rest % a.n_chunks;
  const int ot = rest / a.n_chunks;
  x.o0 = ot * kTileN;
  x.i0 = it * kRowTile;
  x.k0 = x.chunk * kKChunk;
  x.k_len = min(a.K, x.k0 + kKChunk) - x.k0;
  x.n_steps = (x.k_len + kStep - 1) / kStep;
  x.out_tile = ot * a.n_itiles + it;
  return x;
}

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

// The activation producer (one thread of warp 5) first waits for the previous
// kernel on the stream, which writes the rounded activations, then keeps the
// 2-deep activation ring full over the CTA's whole tile sequence.
__device__ void producer_x(const Ctx& c, const MmArgs& a, const CUtensorMap* tm_x) {
  wait_prior_grid();
  int g = 0;
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile x = tile_of(a, t);
    for (int j = 0; j < x.n_steps; ++j, ++g) {
      const int s = g % kXStages;
      if (g >= kXStages && !wait_bar(c, kEmpty0 + s, ((g / kXStages) - 1) & 1)) {
        t = a.n_tiles;
        break;
      }
      const int regions = min(kStep, x.k_len - j * kStep) / kRegion;  // 1 .. 4
      mbar_arrive_expect_tx(bar_addr(c, kFull0 + s), regions * kXRegionBytes);
      for (int rg = 0; rg < regions; ++rg)
        tma_load_2d(c.sbase + kXOff + s * kXBytes + rg * kXRegionBytes, tm_x,
                    x.k0 + j * kStep + rg * kRegion, x.i0, bar_addr(c, kFull0 + s));
    }
  }
  // Copies still in flight must land before the CTA's shared memory goes away
  // (normally the MMA thread has waited for every one already).
  for (int s = 0; s < kXStages; ++s) {
    const int last = g - 1 - ((g - 1 - s) % kXStages + kXStages) % kXStages;
    if (last >= 0 && !mbar_wait(bar_addr(c, kFull0 + s), (last / kXStages) & 1))
      set_error(c.hdr, DA_DEVERR_TIMEOUT);
  }
}

// Tiles alternate between the two accumulators; an accumulator is reused once
// the epilogue has read it.  One wait and one commit per step.  Returns the
// number of steps whose MMAs were issued and committed.
__device__ int mma_issuer(const Ctx& c, const MmArgs& a, uint32_t tmem) {
  const uint64_t a_desc0 = umma::smem_desc(c.sbase + kAOff, 16, 1024, umma::kSwizzle128B);
  const uint64_t b_desc0 = umma::smem_desc(c.sbase + kXOff, 16, 1024, umma::kSwizzle128B);
  int g = 0, k = 0;
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++k) {
    const Tile x = tile_of(a, t);
    const int tb = k & 1;
    if (k >= 2 && !wait_bar(c, kDEmpty0 + tb, ((k >> 1) - 1) & 1)) return g;
    umma::fence_after_sync();
    const uint32_t d = tmem + tb * kRowTile;
    for (int j = 0; j < x.n_steps; ++j, ++g) {
      const int sx = g % kXStages, sa = g % kAStages;
      if (!wait_bar(c, kFull0 + sx, (g / kXStages) & 1)) return g;
      umma::fence_after_sync();
      const int n_mma = min(kStep, x.k_len - j * kStep) / 16;  // 4 .. 16
      // descriptors of this step's operands; each MMA adds a constant offset
      // (K = 16 is 32 bytes of a 128-byte region row; the start address field
      // holds bytes / 16 and never carries out at these offsets)
      const uint64_t ad0 = a_desc0 + (uint64_t)(sa * (kABytes >> 4));
      const uint64_t bd0 = b_desc0 + (uint64_t)(sx * (kXBytes >> 4));
      umma::mma_bf16(d, ad0, bd0, kIdesc, j ? 1u : 0u);
#pragma unroll
      for (int kk = 1; kk < kStep / 16; ++kk) {
        if (kk < n_mma)
          umma::mma_bf16(d, ad0 + (uint64_t)(((kk / 4) * kARegionBytes + (kk % 4) * 32) >> 4),
                         bd0 + (uint64_t)(((kk / 4) * kXRegionBytes + (kk % 4) * 32) >> 4), kIdesc,
                         1u);
      }
      umma::commit(bar_addr(c, kEmpty0 + sx));
    }
    umma::commit(bar_addr(c, kDFull0 + tb));
  }
  return g;
}

// The arrive of a tcgen05.commit lands some time after the MMAs it tracks;
// before the CTA's shared memory is handed on, the last arrive on every ring
// slot's release barrier must have landed.
__device__ void drain_commits(const Ctx& c, int n_done) {
  for (int s = 0; s < kXStages; ++s) {
    const int last = n_done - 1 - ((n_done - 1 - s) % kXStages + kXStages) % kXStages;
    if (last >= 0 && !mbar_wait(bar_addr(c, kEmpty0 + s), (last / kXStages) & 1))
      set_error(c.hdr, DA_DEVERR_TIMEOUT);
  }
}

// Dequantizing warp d (0..15) covers weight rows 8d .. 8d + 7 of the tile; lane
// l takes row 8d + l / 4 and, in each 128-wide half h of every step, blocks
// 2 (l % 4), 2 (l % 4) + 1 (weights 128 h + 32 (l % 4) .. +31).  For each half
// a thread fetches its own 16 bytes of codes and the 4-byte word of block
// scales holding its two blocks with cp.async, kRawStages - 1 steps ahead,
// into a ring only it reads, so the weight stream needs no barrier and no
// copy engine.
__device__ void dequant(const Ctx& c, const MmArgs& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = lane & 3;
  const int tid = dq_index(warp) * 32 + lane;
  const int r = dq_index(warp) * 8 + (lane >> 2);
  const bool leader = lane == 0;
  const int G = gridDim.x;
  // lane 0 waits (one mbarrier poll per warp, not 32) and the warp follows:
  // every lane takes the same branch
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (leader) ok = wait_bar(c, bar, parity) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
  };
  // prefetch cursor over the CTA's steps
  int tf = blockIdx.x, jf = 0, gf = 0;
  Tile xf = tile_of(a, tf);
  auto prefetch = [&]() {
    if (tf < a.n_tiles) {
      const int slot = gf % kRawStages;
      const size_t row = (size_t)(xf.o0 + r);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kb = jf * kStep + h * kSub;  // K of the half step within the chunk
        if (kb + 32 * q < xf.k_len) {  // weights past the end of K are never fetched
          cp_async16(c.sbase + kRawOff + slot * kRawBytes + tid * 32 + h * 16,
                     a.codes + row * (a.K / 2) + (xf.k0 + kb) / 2 + 16 * q);
          cp_async4(c.sbase + kSOff + slot * kSBytes + tid * 8 + h * 4,
                    a.scales + row * (a.K / 16) + (xf.k0 + kb) / 16 + 4 * (q >> 1));
        }
      }
      ++gf;
      if (++jf == xf.n_steps) {
        jf = 0;
        tf += G;
        if (tf < a.n_tiles) xf = tile_of(a, tf);
      }
    }
    cp_async_commit();  // one group per step, empty past the last step
  };
  for (int i = 0; i < kRawStages - 1; ++i) prefetch();
  bool ok = true;
  int g = 0;
  for (int t = blockIdx.x; t < a.n_tiles && ok; t += G) {
    const Tile x = tile_of(a, t);
    for (int j = 0; j < x.n_steps; ++j, ++g) {
      prefetch();                       // step g + kRawStages - 1
      cp_async_wait<kRawStages - 1>();  // this thread's copies of step g have landed
      const int slot = g % kRawStages, sa = g % kAStages, sx = g % kXStages;
      // the weight slot is free once the MMAs of step g - kAStages are done
      if (g >= kAStages &&
          !wait_w(kEmpty0 + (g - kAStages) % kXStages, ((g - kAStages) / kXStages) & 1)) {
        ok = false;
        break;
      }
      bool wrote = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // half step h: K 128 h .. 128 h + 127 of the step
        const bool live = j * kStep + h * kSub + 32 * q < x.k_len;
        if (!live) continue;
        const uint4 w = *reinterpret_cast<const uint4*>(c.smem + kRawOff + slot * kRawBytes +
                                                       tid * 32 + h * 16);
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(c.smem + kSOff + slot * kSBytes +
                                                               tid * 8 + h * 4);
        // the two blocks' scales (bytes 2 (q & 1), +1 of the word) as f16 pairs (s, s)
        const uint32_t s2 = e4m3x2_to_f16x2((q & 1) ? sw >> 16 : sw & 0xffffu);
        const uint32_t sc0 = __byte_perm(s2, 0, 0x1010), sc1 = __byte_perm(s2, 0, 0x3232);
        uint8_t* arow = c.smem + kAOff + sa * kABytes + (2 * h + (q >> 1)) * kARegionBytes +
                        r * 128;
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // 16-byte chunk 4 (q & 1) + e of the region row
          uint32_t hv[4], o[4];
          e2m1x8_to_f16x2(words[e], hv);
#pragma unroll
          for (int u = 0; u < 4; ++u) o[u] = f16x2_to_bf16x2(hmul2(hv[u], e < 2 ? sc0 : sc1));
          *reinterpret_cast<uint4*>(arow + (((4 * (q & 1) + e) ^ (r & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
        wrote = true;
      }
      if (wrote) fence_proxy_async();
      __syncwarp();
      if (leader) mbar_arrive(bar_addr(c, kFull0 + sx));
    }
  }
  cp_async_wait<0>();  // none of this thread's copies may still be in flight at exit
}

// Warps 21-24: thread r = weight row r of the tile = tensor-memory lane r
// (warp w reads lanes 32 (w % 4) ..).
__device__ void epilogue(const Ctx& c, const MmArgs& a, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const bool leader = lane == 0;
  const bool elected = threadIdx.x == kEpWarp0 * 32;
  volatile int* last = reinterpret_cast<volatile int*>(c.smem + kLastSlot);
  const size_t cstride = (size_t)a.n * a.N;  // between chunks of the partials
  bool ok = true;
  int k = 0;
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++k) {
    const Tile x = tile_of(a, t);
    const int tb = k & 1;
    if (ok) {
      int w_ok = 1;
      if (leader) w_ok = wait_bar(c, kDFull0 + tb, (k >> 1) & 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w_ok, 0) != 0;
    }
    if (named_bar_or(kEpBarrier, kEpThreads, !ok)) break;
    umma::fence_after_sync();
    float v[32];
    umma::ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + tb * kRowTile, v);
    umma::wait_ld();
    umma::fence_before_sync();
    __syncwarp();
    if (leader) mbar_arrive(bar_addr(c, kDEmpty0 + tb));  // the MMAs may refill it
    const int o = x.o0 + r;
    const int rows = min(kRowTile, a.n - x.i0);
    if (a.n_chunks == 1) {
#pragma unroll
      for (int i = 0; i < kRowTile; ++i) {
        if (i < rows) {
          const float yv = a.global_scale * v[i];
          a.y[(size_t)(x.i0 + i) * a.N + o] = yv;
          if (a.y_bf16) a.y_bf16[(size_t)(x.i0 + i) * a.N + o] = __float2bfloat16_rn(yv);
        }
      }
      continue;
    }
    float* mine = a.part + x.chunk * cstride + (size_t)x.i0 * a.N + o;
#pragma unroll
    for (int i = 0; i < kRowTile; ++i)
      if (i < rows) mine[(size_t)i * a.N] = v[i];
    // The last chunk CTA of this output tile to get here adds all partials in
    // chunk order.
    __threadfence();
    named_bar_sync(kEpBarrier, kEpThreads);
    if (elected) *last = atomicAdd(a.tile_count + x.out_tile, 1) == a.n_chunks - 1;
    named_bar_sync(kEpBarrier, kEpThreads);
    if (!*last) continue;
    __threadfence();
    // sum = P_0, then sum += P_c for c = 1, 2, ...: all 32 rows of a chunk are
    // loaded before they are added, so the loads overlap
    const float* p0 = a.part + (size_t)x.i0 * a.N + o;
#pragma unroll
    for (int i = 0; i < kRowTile; ++i) v[i] = (i < rows) ? __ldcg(p0 + (size_t)i * a.N) : 0.f;
    for (int ch = 1; ch < a.n_chunks; ++ch) {
      const float* pc = p0 + ch * cstride;
      float u[kRowTile];
#pragma unroll
      for (int i = 0; i < kRowTile; ++i) u[i] = (i < rows) ? __ldcg(pc + (size_t)i * a.N) : 0.f;
#pragma unroll
      for (int i = 0; i < kRowTile; ++i) v[i] += u[i];
    }
#pragma unroll
    for (int i = 0; i < kRowTile; ++i) {
      if (i < rows) {
        const float yv = a.global_scale * v[i];
        a.y[(size_t)(x.i0 + i) * a.N + o] = yv;
        if (a.y_bf16) a.y_bf16[(size_t)(x.i0 + i) * a.N + o] = __float2bfloat16_rn(yv);
      }
    }
    if (elected) a.tile_count[x.out_tile] = 0;  // ready for the next call
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_mm_kernel(MmArgs a, const __grid_constant__ CUtensorMap tm_x) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
  c.hdr = a.hdr;
  const int warp = threadIdx.x >> 5;
  allow_next_grid();  // the next call's first kernel may be scheduled; it waits for this grid
  if (c.sbase & 1023u) {  // the swizzled layouts need 1024-byte-aligned shared memory
    if (threadIdx.x == 0) set_error(a.hdr, DA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;  // TMA expect_tx arrive or tcgen05.commit
      if (i >= kFull0 && i < kFull0 + kXStages) count = kDqWarps + 1;  // + the activation copy
      if (i == kDEmpty0 || i == kDEmpty0 + 1) count = kEpWarps;
      mbar_init(bar_addr(c, i), count);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(c.sbase + kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

  int n_done = 0;  // steps the MMA thread committed
  if (warp == kXWarp) {
    if ((threadIdx.x & 31) == 0) producer_x(c, a, &tm_x);
  } else if (warp == kMmaWarp) {
    if ((threadIdx.x & 31) == 0) {
      n_done = mma_issuer(c, a, tmem);
      umma::commit(bar_addr(c, kDrain));  // arrives once every MMA above has completed
    }
  } else if (warp >= kEpWarp0) {
    // Its stores come after the MMAs, which come after the producer's wait
    // for the previous kernel: they never overtake that kernel's accesses.
    epilogue(c, a, tmem);
  } else if (is_dq_warp(warp)) {
    dequant(c, a);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    umma::fence_after_sync();
    if ((threadIdx.x & 31) == 0) {
      if (!mbar_wait(bar_addr(c, kDrain), 0)) set_error(a.hdr, DA_DEVERR_TIMEOUT);
      drain_commits(c, n_done);
    }
    __syncwarp();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// fp32 / bf16 activations [n, K] -> bf16 [n_pad, K] (round to nearest even),
// rows n .. n_pad - 1 zero, eight elements per thread and step; also clears
// the call's error word and the per-tile chunk counters.
__global__ void nvfp4_round_kernel(const void* x, int x_dtype, __nv_bfloat16* xr, int32_t* hdr,
                                   int32_t* tile_count, int n_tiles, int n, int n_pad, int K) {
  wait_prior_grid();
  allow_next_grid();  // after the wait: the next kernel may read the weight early
  const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  if (tid == 0) hdr[kHdrError] = 0;  // errors of this call only
  for (size_t t = tid; t < (size_t)n_tiles; t += nthreads) tile_count[t] = 0;
  const size_t total = (size_t)n_pad * K / 8, valid = (size_t)n * K / 8;
  for (size_t v = tid; v < total; v += nthreads) {
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

// Multiprocessors of the current device (cached per device).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev >= 64) {
    int v = 0;
    return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 0;
  }
  if (cache[dev] == 0 &&
      cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    cache[dev] = 0;
  return cache[dev];
}

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

int n_chunks_of(int K) { return (K + kKChunk - 1) / kKChunk; }

size_t xr_bytes(int n, int K) { return round_up((size_t)round_up(n, kRowTile) * K * 2, 256); }

int n_tiles_of(int n, int N) { return (N / kTileN) * (int)(round_up(n, kRowTile) / kRowTile); }

size_t counter_bytes(int n, int N) { return round_up((size_t)n_tiles_of(n, N) * 4, 256); }

bool shape_ok(int n, int N, int K) {
  if (n < 0 || N <= 0 || K <= 0 || N % kTileN || K % kRegion) return false;
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
  size_t b = kHdr + counter_bytes(n, N) + xr_bytes(n, K);
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
  int32_t* tile_count = reinterpret_cast<int32_t*>(base + kHdr);
  __nv_bfloat16* xr = reinterpret_cast<__nv_bfloat16*>(base + kHdr + counter_bytes(n, N));
  float* part = nc > 1 ? reinterpret_cast<float*>(base + kHdr + counter_bytes(n, N) +
                                                  xr_bytes(n, K))
                       : nullptr;

  alignas(64) CUtensorMap tm_x;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)n_pad};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {kRegion, kRowTile};
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
  a.codes = codes;
  a.scales = scales;
  a.part = part;
  a.y = y;
  a.y_bf16 = static_cast<__nv_bfloat16*>(y_bf16);
  a.hdr = static_cast<int32_t*>(ws);
  a.tile_count = tile_count;
  a.global_scale = global_scale;
  a.n = n;
  a.N = N;
  a.K = K;
  a.n_chunks = nc;
  a.n_itiles = n_pad / kRowTile;

  const size_t vec = (size_t)n_pad * K / 8;
  const int round_blocks = (int)std::min<size_t>((vec + 255) / 256, 4096);
  if (launch_after(nvfp4_round_kernel, dim3(round_blocks), dim3(256), 0, st, x, (int)x_dtype, xr,
                   a.hdr, tile_count, n_tiles_of(n, N), (int)n, n_pad, (int)K) != cudaSuccess)
    return DA_ERR_CUDA;
  const long long tiles = (long long)(N / kTileN) * nc * a.n_itiles;
  if (tiles >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
  a.n_tiles = (int)tiles;
  const int sms = sm_count();
  if (sms <= 0) return DA_ERR_CUDA;
  const int grid = (int)std::min<long long>(tiles, sms);  // persistent: one CTA per SM
  if (launch_after(nvfp4_mm_kernel, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, st, a, tm_x) != cudaSuccess)
    return DA_ERR_CUDA;
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
