// Split kernel, tensor-core variant: up to 128 query heads sharing one latent
// KV row of 576 dims whose first 512 dims are the value (MLA-style sparse
// decode, the case "Sparse MLA decode is not batch-invariant" -- FlashMLA
// issue #212 -- reports on).
//
// Both contractions run on tcgen05 tensor cores with fp32 accumulators in
// tensor memory (TMEM):
//     S = Q K^T      M = 128 heads, N = 32 entries, K = 576   (36 MMAs of K=16)
//     O += P V_half  M = 128 heads, N = 256 dims,   K = 32    (2 MMAs)
// O for 128 heads x 512 dims in fp32 would fill all of one SM's tensor memory,
// so a (row, split) item runs as two units, one per half of the value dims;
// each unit computes the full S itself (the same instructions on the same
// data, so both halves see the same bits).
//
// Operand placement.  The first 384 dims of Q live in TMEM (192 columns) and
// feed 24 of the 36 S MMAs as the A operand, so those read only the K tile
// from shared memory; dims 384..575 of Q stay in shared memory (48 KB).  TMEM
// columns: Q [0,192), S as two K-half partial accumulators [192,224) and
// [224,256) (two independent MMA chains), O [256,512).
// Shared memory: Q tail, four 32-entry KV stages (36 KB each), P (8 KB).
//
// Roles inside a CTA (288 threads):
//   warps 0-3  softmax: thread i owns head i = TMEM lane i.  It loads its row
//              of Q into TMEM at the start of a unit, reads its row of S,
//              keeps the running max and sum in fp32, writes P (bf16) into
//              shared memory and rescales its row of O when the max it uses
//              moves by more than 2^8.
//   warps 4-7  producer: gathers each entry's 1152-byte latent row with
//              16-byte cp.async into the 128-byte-swizzled K-major layout the
//              tensor core reads (and the unit's Q tail at its start).
//   warp 8     MMA issue (one thread) and TMEM allocation.
// Every wait on an mbarrier is bounded; on time-out the kernel records
// DA_DEVERR_TIMEOUT, every role leaves its loop, outstanding tensor-core work
// is drained (bounded) and TMEM is freed.
#include "common.cuh"
#include "tcgen05.cuh"

namespace da {
namespace {

constexpr int kHeads = 128;       // MMA M (query heads, zero-padded)
constexpr int kDqk = 576;
constexpr int kDvHalf = 256;      // value dims per unit
constexpr int kSub = 64;          // entries per sub-tile (MMA N of S, K of P.V)
constexpr int kRegions = kDqk / 64;  // 64-dim swizzle regions of a row
constexpr int kRowChunks = kDqk / 8; // 16-byte chunks of a row (72)
constexpr int kQT = 384;          // dims of Q held in TMEM (A operand)
constexpr int kQTCols = kQT / 2;  // 192 TMEM columns (two bf16 per column)
constexpr int kQSRegions = (kDqk - kQT) / 64;  // 3 smem regions of Q (dims 384..575)
constexpr int kStages = 2;

// shared memory map (bytes)
constexpr int kQSBytes = kQSRegions * kHeads * 128;        // 49152
constexpr int kStageRegion = kSub * 128;                    // 8192
constexpr int kStageBytes = kRegions * kStageRegion;        // 73728
constexpr int kStageOffset = kQSBytes;
constexpr int kPOffset = kStageOffset + kStages * kStageBytes;  // 196608
constexpr int kPBytes = kHeads * kSub * 2;                  // 16384 (128-byte swizzle)
constexpr int kBarOffset = kPOffset + kPBytes;              // 212992
enum { kFull0 = 0, kEmpty0 = kFull0 + kStages, kSFull = kEmpty0 + kStages, kSFree, kPFull,
       kODone, kOFree, kQFull, kQTFull, kQFree, kDrain, kNumBars };
constexpr int kTmemSlot = kBarOffset + kNumBars * 8;
static_assert(kPOffset % 1024 == 0 && kStageOffset % 1024 == 0, "swizzle atoms 1024-aligned");
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kSmemBytes = kAbortSlot + 12;
static_assert(kSmemBytes <= 232448, "fits the 227 KB per-block limit");

constexpr int kThreads = 288;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = kQTCols;  // S partial accumulators at [192, 256)
constexpr int kKSteps = kDqk / 16;   // 36 MMAs of K = 16 per S tile
constexpr int kEntPerWarp = kSub / 4;  // entries each producer warp gathers
constexpr uint32_t kOCol = 256;      // O accumulator columns [256, 512)
constexpr float kRescaleLog2 = 8.f;

constexpr uint32_t kIdescS = umma::idesc_bf16_f32(kHeads, kSub, false);
constexpr uint32_t kIdescO = umma::idesc_bf16_f32(kHeads, kDvHalf, true);

__device__ __forceinline__ void cp_async16_zero(uint32_t dst, const void* any_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(dst), "l"(any_src)
               : "memory");
}

// The mbarrier receives one arrive once all earlier cp.async of this thread land.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;  // shared address of smem[0]
  volatile int* abort_flag;
  int32_t* hdr;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) {
  return c.sbase + kBarOffset + 8 * i;
}

// Bounded wait that also gives up when the abort flag is raised.
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

// A unit: one half of the value dims of one (row, split) item.
struct MlaUnit {
  int slot, b, half, t_begin, t_end;  // entry range [t_begin, t_end)
  int l_main;                         // entries before the second source starts
  bool single, empty;
};

__device__ __forceinline__ MlaUnit mla_unit(const Launch& p, int u) {
  const int4 d = __ldg(reinterpret_cast<const int4*>(p.item_desc) + (u >> 1));
  MlaUnit x;
  x.single = d.x < 0;
  x.slot = x.single ? ~d.x : d.x;
  x.b = x.slot / p.max_splits;
  x.half = u & 1;
  x.t_begin = d.y * kMlaTile;
  x.t_end = min(d.z * kMlaTile, d.w);
  x.empty = x.t_end <= x.t_begin;
  x.l_main = p.extra_k ? clamp_len(__ldg(p.lengths + x.b), p.capacity) : 0x7fffffff;
  return x;
}

// Latent-cache row holding entry `tok` of row b (H_kv = 1); entries from
// l_main on come from the second source (*src = 1).
__device__ __forceinline__ bool latent_row(const Launch& p, int b, int tok, int l_main,
                                           long long* row, int* src) {
  *src = 0;
  if (tok >= l_main) {
    const int slot = __ldg(p.extra_table + (size_t)b * p.extra_width + (tok - l_main));
    *row = slot;
    *src = 1;
    return slot >= 0 && slot < p.extra_num_blocks;
  }
  if (p.layout == DA_KV_CONTIGUOUS) {
    *row = (long long)b * p.width + tok;
    return true;
  }
  if (p.layout == DA_KV_PAGED) {
    const int page = __ldg(p.table + (size_t)b * p.width + tok / p.page_size);
    *row = (long long)page * p.page_size + tok % p.page_size;
    return page >= 0 && page < p.num_blocks;
  }
  const int slot = __ldg(p.table + (size_t)b * p.width + tok);
  *row = slot;
  return slot >= 0 && slot < p.num_blocks;
}

// 128-byte swizzle inside a 1024-byte-aligned region of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------- producer
__device__ void producer(const Launch& p, const Ctx& c, int n_units) {
  const int pt = threadIdx.x - 128;  // 0..127
  const int pw = pt >> 5, pl = pt & 31;
  uint32_t g = 0, n_ne = 0;
  bool alive = true;
  bool bad = false;
  for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
    const MlaUnit x = mla_unit(p, u);
    if (x.empty) continue;
    // Q dims 384..575 of row b (zero rows past H_q) into shared memory, once
    // the previous unit's S MMAs are done
    if (!wait_bar(c, kQFree, (n_ne & 1) ^ 1)) break;
    for (int i = 0; i < kHeads * (kQSRegions * 8) / 128; ++i) {
      const int q = pt + 128 * i;
      const int r = q / (kQSRegions * 8), j = q % (kQSRegions * 8);
      const uint32_t dst = c.sbase + (j >> 3) * (kHeads * 128) + sw128(r, j & 7);
      if (r < p.H_q)
        cp_async16(dst, p.q + ((size_t)x.b * p.H_q + r) * kDqk + kQT + j * 8);
      else
        cp_async16_zero(dst, p.q);
    }
    cp_async_arrive_noinc(bar_addr(c, kQFull));
    // warm L2 with the next unit's query rows (its softmax warps load them
    // into tensor memory at its start)
    if (u + (int)gridDim.x < n_units) {
      const MlaUnit nx = mla_unit(p, u + gridDim.x);
      const char* qn = reinterpret_cast<const char*>(p.q + (size_t)nx.b * p.H_q * kDqk);
      const int lines = min(p.H_q, kHeads) * kDqk * 2 / 128;
      for (int i = pt; i < lines; i += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + (size_t)i * 128));
    }
    // lanes 0-7 of producer warp pw look up the rows of entries 8*pw .. 8*pw+7
    // of a sub-tile; the lookup for the next sub-tile is issued before the
    // copies of the current one so its latency hides behind them
    // ok: 0 = masked / bad index, 1 = main source, 2 = second source
    auto lookup = [&](int t0, long long& row, int& ok) {
      row = 0;
      ok = 0;
      const int e = kEntPerWarp * pw + pl;
      if (pl < kEntPerWarp && t0 + e < x.t_end) {
        int src;
        const bool good = latent_row(p, x.b, t0 + e, x.l_main, &row, &src);
        ok = good ? 1 + src : 0;
        bad |= !good;
      }
    };
    long long nx_row;
    int nx_ok;
    lookup(x.t_begin, nx_row, nx_ok);
    for (int t0 = x.t_begin; t0 < x.t_end; t0 += kSub, ++g) {
      const int stage = g % kStages;
      if (!wait_bar(c, kEmpty0 + stage, ((g / kStages) & 1) ^ 1)) {
        alive = false;
        break;
      }
      const uint32_t sb = c.sbase + kStageOffset + stage * kStageBytes;
      const long long my_row = nx_row;
      const int my_ok = nx_ok;
      if (t0 + kSub < x.t_end) lookup(t0 + kSub, nx_row, nx_ok);
#pragma unroll 4
      for (int i = 0; i < kEntPerWarp * kRowChunks / 32; ++i) {
        const int q = pl + 32 * i;
        const int e = q / kRowChunks, j = q % kRowChunks;
        const long long row = __shfl_sync(0xffffffffu, my_row, e);
        const int ok = __shfl_sync(0xffffffffu, my_ok, e);
        const uint32_t dst = sb + (j >> 3) * kStageRegion + sw128(kEntPerWarp * pw + e, j & 7);
        if (ok)
          cp_async16(dst, (ok == 1 ? p.k : p.extra_k) + (size_t)row * kDqk + j * 8);
        else
          cp_async16_zero(dst, p.k);  // masked entries read as zeros, never garbage
      }
      cp_async_arrive_noinc(bar_addr(c, kFull0 + stage));
    }
    ++n_ne;
  }
  if (bad) set_error(p.hdr, DA_DEVERR_INDEX);
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- MMA issue
__device__ void mma_issuer(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  uint32_t g = 0, n_ne = 0;
  // base descriptors; per-MMA ones differ only by a constant start offset
  const uint64_t b_stage0 =  // K tile, K-major, 128-byte swizzle
      umma::smem_desc(c.sbase + kStageOffset, 16, 1024, umma::kSwizzle128B);
  const uint64_t a_q0 =      // Q tail, K-major, 128-byte swizzle
      umma::smem_desc(c.sbase, 16, 1024, umma::kSwizzle128B);
  const uint64_t a_p0 =      // P, K-major, 128-byte swizzle
      umma::smem_desc(c.sbase + kPOffset, 16, 1024, umma::kSwizzle128B);
  const uint64_t b_v0 =      // V = leading dims of the K tile, MN-major
      umma::smem_desc(c.sbase + kStageOffset, kStageRegion, 1024, umma::kSwizzle128B);
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const MlaUnit x = mla_unit(p, u);
    if (x.empty) continue;
    const int n_sub = (x.t_end - x.t_begin + kSub - 1) / kSub;
    if (!wait_bar(c, kQFull, n_ne & 1)) return;   // Q tail in shared memory
    fence_proxy_async();
    if (!wait_bar(c, kQTFull, n_ne & 1)) return;  // Q head dims in TMEM
    umma::fence_after_sync();
    auto pv = [&](uint32_t gp, bool first) -> bool {
      if (!wait_bar(c, kPFull, gp & 1)) return false;
      if (first && !wait_bar(c, kOFree, (n_ne & 1) ^ 1)) return false;
      umma::fence_after_sync();
      const uint64_t bv = b_v0 + (uint64_t)(((gp % kStages) * kStageBytes +
                                             4 * x.half * kStageRegion) >> 4);
#pragma unroll
      for (int kk = 0; kk < kSub / 16; ++kk)
        umma::mma_bf16(tmem + kOCol, a_p0 + (uint64_t)((kk * 32) >> 4),
                       bv + (uint64_t)((kk * 2048) >> 4), kIdescO,
                       (first && kk == 0) ? 0u : 1u);
      umma::commit(bar_addr(c, kODone));
      umma::commit(bar_addr(c, kEmpty0 + (gp % kStages)));
      return true;
    };
    // Issue order PV(g-1), S(g): the PV that frees stage g-1 is queued before
    // the S of tile g, so the producer refills that stage while S(g) runs.
    for (int i = 0; i < n_sub; ++i, ++g) {
      if (i > 0 && !pv(g - 1, i == 1)) return;
      const int stage = g % kStages;
      if (!wait_bar(c, kFull0 + stage, (g / kStages) & 1)) return;
      fence_proxy_async();
      if (!wait_bar(c, kSFree, (g & 1) ^ 1)) return;  // softmax has read S(g-1)
      umma::fence_after_sync();
      // S = Q K^T: 36 MMAs of M = 128, N = 64, K = 16 into columns [192, 256)
      const uint64_t b0 = b_stage0 + (uint64_t)((stage * kStageBytes) >> 4);
      const uint32_t d_s = tmem + kSCol;
#pragma unroll
      for (int k = 0; k < kKSteps; ++k) {  // K step k: dims 16k .. 16k+15
        const uint64_t b = b0 + (uint64_t)(((k / 4) * kStageRegion + (k % 4) * 32) >> 4);
        if (k < kQT / 16)  // A = Q rows in TMEM (8 columns per 16 dims)
          umma::mma_bf16_ta(d_s, tmem + k * 8, b, kIdescS, k ? 1u : 0u);
        else               // A = Q tail in shared memory
          umma::mma_bf16(d_s, a_q0 + (uint64_t)((((k - kQT / 16) / 4) * kHeads * 128 +
                                                   (k % 4) * 32) >> 4),
                         b, kIdescS, 1u);
      }
      umma::commit(bar_addr(c, kSFull));
      if (i == n_sub - 1) umma::commit(bar_addr(c, kQFree));
    }
    if (!pv(g - 1, n_sub == 1)) return;
    ++n_ne;
  }
}

// ---------------------------------------------------------------- softmax + epilogue
__device__ void softmax_warps(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = threadIdx.x;  // head = tensor-memory lane
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  uint32_t g = 0, n_ne = 0;
  // warp-uniform bounded wait (lane 0 waits, everyone follows its verdict)
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto arrive_w = [&](int bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, bar));
  };
  // Q dims 0..383 of head `row` of row b into TMEM columns [0, 192): two bf16
  // per column, the lower dim in the low half; then signal the MMA thread.
  auto load_q = [&](int b) {
    const bool ok = row < p.H_q;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.H_q + row) * kDqk);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      uint4 w[24];
#pragma unroll
      for (int i = 0; i < 24; ++i) w[i] = ok ? __ldg(qrow + half * 24 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int ch = 0; ch < 3; ++ch) {
        uint32_t r32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          r32[4 * i + 0] = w[ch * 8 + i].x;
          r32[4 * i + 1] = w[ch * 8 + i].y;
          r32[4 * i + 2] = w[ch * 8 + i].z;
          r32[4 * i + 3] = w[ch * 8 + i].w;
        }
        umma::st_32x32b_x32_u(lane_base + (half * 3 + ch) * 32, r32);
      }
    }
    umma::wait_st();
    umma::fence_before_sync();
    arrive_w(kQTFull);
  };
  bool q_ready = false;  // Q of the coming unit already in TMEM
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const MlaUnit x = mla_unit(p, u);
    const bool head_ok = row < p.H_q;
    const size_t out_row = ((size_t)x.b * p.H_q + row) * 512 + x.half * kDvHalf;
    if (x.empty) {  // empty row: out = 0, lse = -inf (always a single split)
      if (head_ok) {
        for (int d = 0; d < kDvHalf; ++d) p.out[out_row + d] = __float2bfloat16_rn(0.f);
        if (x.half == 0) p.lse[(size_t)x.b * p.H_q + row] = -INFINITY;
      }
      continue;
    }
    const int n_sub = (x.t_end - x.t_begin + kSub - 1) / kSub;
    if (!q_ready) {
      // (first unit only: later units get their Q while the previous unit's
      // epilogue is still ahead, see below)
      if (!wait_w(kQFree, (n_ne & 1) ^ 1)) return;
      umma::fence_after_sync();
      load_q(x.b);
    }
    q_ready = false;
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < n_sub; ++i, ++g) {
      if (!wait_w(kSFull, g & 1)) return;
      umma::fence_after_sync();
      float s[64];
      {
        float s_hi[32];
        umma::ld_32x32b_x32(lane_base + kSCol, *reinterpret_cast<float(*)[32]>(s));
        umma::ld_32x32b_x32(lane_base + kSCol + 32, s_hi);
        umma::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) s[32 + j] = s_hi[j];
      }
      umma::fence_before_sync();
      arrive_w(kSFree);
      const int n_valid = min(kSub, x.t_end - (x.t_begin + i * kSub));
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kSub; ++j) {
        s[j] = (j < n_valid) ? s[j] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
      // the max used for the exponentials moves only when the tile max
      // exceeds it by more than 2^8 (fewer O rescales; P stays <= 256)
      const float m_new = (i == 0 || mt > m_used + kRescaleLog2) ? mt : m_used;
      const float alpha = (i == 0) ? 1.f : ex2(m_used - m_new);
      float sum = 0.f;
      uint32_t pk[kSub / 2];
#pragma unroll
      for (int j = 0; j < kSub; j += 2) {
        const float p0 = ex2(s[j] - m_new), p1 = ex2(s[j + 1] - m_new);
        sum += p0;
        sum += p1;
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l = (i == 0) ? sum : fmaf(l, alpha, sum);
      if (i > 0) {  // PV of the previous sub-tile must be done with P and O
        if (!wait_w(kODone, (g - 1) & 1)) return;
        umma::fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int ch = 0; ch < kDvHalf / 32; ++ch) {
            float o[32];
            umma::ld_32x32b_x32(lane_base + kOCol + ch * 32, o);
            umma::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= alpha;
            umma::st_32x32b_x32(lane_base + kOCol + ch * 32, o);
          }
          umma::wait_st();
        }
      }
      m_used = m_new;
      // P row (64 bf16 = 128 bytes) into the 128-byte-swizzled K-major tile
      uint8_t* prow = c.smem + kPOffset + row * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(prow + ((cc ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async();
      umma::fence_before_sync();
      arrive_w(kPFull);
      if (i == n_sub - 1) {
        // All S MMAs of this unit are done (S of the last tile was read), so
        // TMEM columns [0, 192) are free: load the next unit's Q now and let
        // the MMA thread start on it while this unit's epilogue runs.
        for (int u2 = u + gridDim.x; u2 < n_units; u2 += gridDim.x) {
          const MlaUnit x2 = mla_unit(p, u2);
          if (x2.empty) continue;
          if (!wait_w(kQFree, n_ne & 1)) return;
          umma::fence_after_sync();
          load_q(x2.b);
          q_ready = true;
          break;
        }
      }
    }
    // epilogue: O / l for this half of the value dims
    if (!wait_w(kODone, (g - 1) & 1)) return;
    umma::fence_after_sync();
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kDvHalf / 32; ++ch) {
      float o[32];
      umma::ld_32x32b_x32(lane_base + kOCol + ch * 32, o);
      umma::wait_ld();
      if (head_ok) {
        if (x.single) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + out_row + ch * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h =
                  __floats2bfloat162_rn(o[v * 8 + 2 * e] * inv, o[v * 8 + 2 * e + 1] * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.o_part + ((size_t)x.slot * p.H_q + row) * 512 + x.half * kDvHalf + ch * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(o[4 * v] * inv, o[4 * v + 1] * inv, o[4 * v + 2] * inv,
                                 o[4 * v + 3] * inv);
        }
      }
    }
    umma::fence_before_sync();
    arrive_w(kOFree);
    ++n_ne;
    if (head_ok && x.half == 0) {
      const float lse2 = (l > 0.f) ? m_used + lg2(l) : -INFINITY;
      if (x.single)
        p.lse[(size_t)x.b * p.H_q + row] = (l > 0.f) ? lse2 * kLn2 : -INFINITY;
      else
        p.lse_part[(size_t)x.slot * p.H_q + row] = lse2;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) split_mla_kernel(Launch p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
  c.hdr = p.hdr;
  const int warp = threadIdx.x >> 5;
  wait_prior_grid();  // the plan kernel's outputs
  allow_next_grid();
  const int n_units = p.hdr[kHdrNWork] * 2;
  if ((int)blockIdx.x >= n_units) return;  // uniform across the CTA
  // the swizzled layouts assume 1024-byte-aligned shared addresses
  if (c.sbase & 1023u) {
    if (threadIdx.x == 0) set_error(p.hdr, DA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;                                           // tcgen05.commit
      if ((i >= kFull0 && i < kFull0 + kStages) || i == kQFull) count = 128;  // producer threads
      if (i == kSFree || i == kPFull || i == kOFree || i == kQTFull)
        count = 4;                                                   // softmax warps
      mbar_init(bar_addr(c, i), count);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    umma::tmem_alloc(c.sbase + kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

  if (warp < 4) {
    softmax_warps(p, c, tmem, n_units);
  } else if (warp < 8) {
    producer(p, c, n_units);
  } else if ((threadIdx.x & 31) == 0) {
    mma_issuer(p, c, tmem, n_units);
    // drain: one more commit; its arrival means every MMA issued before it
    // has completed, so tensor memory can be freed
    umma::commit(bar_addr(c, kDrain));
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    umma::fence_after_sync();
    if ((threadIdx.x & 31) == 0) {
      const uint32_t bar = bar_addr(c, kDrain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, 0)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_error(p.hdr, DA_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool mla_supported(int H_q) { return H_q >= 16 && H_q <= kHeads; }

int mla_ctas_per_sm() { return 1; }

cudaError_t launch_split_mla(const Launch& p, int grid, cudaStream_t stream) {
  static const cudaError_t attr = cudaFuncSetAttribute(
      split_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (attr != cudaSuccess) return attr;
  return launch_after(split_mla_kernel, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, stream,
                      p);
}

}  // namespace da
