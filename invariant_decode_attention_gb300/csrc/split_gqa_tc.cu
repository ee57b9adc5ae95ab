// Split kernel, tensor-core variant for grouped-query attention with a
// separate K and V cache: 16 to 128 query heads per KV head, head dim 128,
// bf16, E4M3 or NVFP4 caches.
//
// One unit of work = (row b, split s, KV head h).  Both contractions run on
// tcgen05 tensor cores with fp32 accumulators in tensor memory (TMEM):
//     S = Q K^T      M = 128, N = 64 entries, K = 128 dims   (8 MMAs of K=16)
//     O += P V       M = 128, N = 128 dims,   K = 64 entries (4 MMAs of K=16)
// The G query heads of the group, padded to gp = the power of two >= G (at
// least 16), fill the 128 MMA rows as R = 128 / gp copies; rows past the
// group compute on whatever the Q buffer holds there and are never written
// (a row of an MMA result depends only on its own row of A).  Copy c of the
// group takes entries [c * 64 / R, (c + 1) * 64 / R) of every tile in the
// softmax: a thread owns one (head, copy) row -- one TMEM lane -- with its
// own running max and sum, P is zero outside its copy's entries, and the
// epilogue merges the R copies' (O, max, sum) of each head.  The reference
// value of a row's exponentials moves only when a score exceeds it by more
// than 2^8 (then its O row is rescaled in TMEM), a decision that depends only
// on the unit's own scores.
//
// Memory.  Shared: six 64-entry stages of K and V (bf16 cache; three for a
// quantized cache, plus its raw stages), each tile in the 128-byte-swizzled
// layout the tensor core reads (two 64-dim regions of 64 rows x 128 bytes).
// P of a tile (128 heads x 64 entries, 16-bit) is written over its stage's K
// tile once S has read it.  TMEM: two S buffers, two O accumulators (the
// next unit's first P.V does not wait for the previous unit's epilogue) and
// two Q buffers (the S MMAs' A operand; the next unit's Q is written while
// the current one runs).
//
// Loads (TMA).  For a contiguous cache and for pages of a multiple of 16
// entries, each 16-entry group of a tile is 16 consecutive cache rows: one
// box copy of 16 rows x 64 dims per half of the head's row.  Other layouts
// gather four rows per copy (tile::gather4).  Entries past the split's end,
// and entries whose page or slot is out of range, copy cache row 0 instead
// (their scores are masked), so no stage byte is ever uninitialised.
//
// Roles: warps 0-3 softmax; warps 4-7 epilogue (a unit's O merge and output
// while the softmax warps go on with the next unit); warps 8-9 producer (page
// or index lookups ahead of the copies, TMA issue; for a bf16 cache the two
// warps take alternate tiles, so one issues copies while the other waits for
// its next stage; for a quantized cache warp 8 alone); warp 10 the S MMAs
// (one thread) and TMEM allocation; warps 11-14 converter (Q into tensor
// memory; quantized cache: K and V into the operand stages); warp 15 the
// P.V MMAs (one thread).  Every mbarrier wait is bounded; on time-out the
// kernel records DA_DEVERR_TIMEOUT, every role leaves its loop, outstanding
// tensor-core work is drained (bounded) and TMEM is freed.
//
// Softmax attention and its split/merge are the computation "Sparse MLA
// decode is not batch-invariant" (FlashMLA issue #212) reports on; which CTA
// runs a unit never changes what the unit computes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace da {
namespace {

constexpr int kRows = 128;  // MMA M: query heads of the group, padded
constexpr int kD = 128;
constexpr int kT = kTcTile;  // entries per tile
static_assert(kT == 64, "one 128-byte swizzle row of P per head");
constexpr int kRegion = kT * 128;           // 64 rows x 64 dims (16-bit elements)
constexpr int kTileBytes = 2 * kRegion;     // K (or V) of a tile: 16 KB
constexpr int kStageBytes = 2 * kTileBytes;  // K, then V

constexpr int kMaxStages = 6;     // operand stages
constexpr int kMaxRawStages = 8;  // raw stages (quantized caches)
enum {
  kFull0 = 0, kEmpty0 = kFull0 + kMaxStages,  // operand stages: ready / free
  kRawFull0 = kEmpty0 + kMaxStages,           // quantized cache: copies landed
  kRawEmpty0 = kRawFull0 + kMaxRawStages,     // quantized cache: converted, reusable
  kQConv0 = kRawEmpty0 + kMaxRawStages,       // Q written to tensor memory
  kQFree0 = kQConv0 + 2,
  // P ready and P.V done: eight slots each (tile g uses slot g % 8, phase
  // g / 8).  The S and P.V MMAs are issued by two threads, so the softmax can
  // run up to kStages - 1 tiles ahead of the P.V thread (S(g) needs stage g's
  // copy, which needs P.V(g - kStages) done); eight slots keep every parity
  // wait within one phase of its barrier.
  kSFull0 = kQFree0 + 2, kSFree0 = kSFull0 + 2, kPFull0 = kSFree0 + 2, kPVDone0 = kPFull0 + 8,
  kODone0 = kPVDone0 + 8, kEpiReady0 = kODone0 + 2, kOFree0 = kEpiReady0 + 2,
  kDrain = kOFree0 + 2,
  kStall,  // never signalled: the time-out test hook waits on it
  kNumBars
};

// Shared-memory map.  KT: 0 bf16 cache, 1 E4M3 (one byte per element), 2
// NVFP4 (E2M1 codes and E4M3 block scales); Q8: a quantized cache (1 or 2).
// Q lives in tensor memory (the converter warps write it there, two buffers),
// so shared memory holds only the cache.  bf16: six operand stages that TMA
// fills directly (192 KB in flight per SM: a stage stays busy from its copy,
// ≈ 3–4k cycles to land, through its S, softmax and P.V).  Quantized: TMA
// copies the cache bytes into raw stages (one producer warp) and the
// converter warpgroup writes them, as f16, into four operand stages (the
// MMAs then run on f16 operands, see the converter).  Five E4M3 raw stages
// keep 80 KB of the cache in flight per SM, six NVFP4 stages 72 KB; measured
// against 3 operand + 7 (E4M3) / 8 (NVFP4) raw stages and 5 + 3 / 4, the
// converter, which waits for a free operand stage, is held up least here.
template <int KT>
struct Lay {
  static constexpr bool Q8 = KT != 0;  // a quantized cache: the f16 converter path
  static constexpr int kStages = Q8 ? 4 : 6;     // operand stages (K, V as 16-bit)
  // Raw stage: E4M3 -- K rows, then V rows, 128 bytes each (16 KB); NVFP4 --
  // K codes, V codes (64 bytes a row), then K and V block scales (16 bytes a
  // row: the scale rows of two neighbouring heads, copied together) in 2 KB
  // each (box copies: 16 rows a copy, rows back to back; gathers: 4 rows a
  // copy into its own 128-byte slot, as a tensor copy's shared destination
  // is 128-byte aligned) (12 KB)
  static constexpr int kRawCodeBytes = KT == 2 ? kT * kD / 2 : kT * kD;  // K (or V) codes of a tile
  static constexpr int kRawScaleBytes = KT == 2 ? (kT / 4) * 128 : 0;    // K (or V) scales
  static constexpr int kRawStageBytes = 2 * kRawCodeBytes + 2 * kRawScaleBytes;
  static constexpr int kRawTxBytes = 2 * kRawCodeBytes + (KT == 2 ? 2 * kT * 16 : 0);  // copied
  static constexpr int kRawStages = KT == 2 ? 6 : Q8 ? 5 : 0;
  static constexpr int kStageOffset = 0;
  static constexpr int kRawOffset = kStageOffset + kStages * kStageBytes;
  static constexpr int kBarOffset = kRawOffset + kRawStages * kRawStageBytes;
  static_assert(kRawStageBytes % 1024 == 0, "raw stages keep 1 KB alignment");
  static constexpr int kTmemSlot = kBarOffset + kNumBars * 8;
  static constexpr int kAbortSlot = kTmemSlot + 4;
  // m and l of every row, per O buffer (softmax -> epilogue), then the
  // epilogue's merge scratch: one 32-column chunk of every row's O (rows
  // padded to 33 floats)
  static constexpr int kMergeOffset = (kAbortSlot + 4 + 15) / 16 * 16;
  static constexpr int kSmemBytes = kMergeOffset + (2 * 2 * kRows + kRows * 33) * 4;
  // warps 0-3 softmax, 4-7 epilogue, 8-9 producer, 10 S MMAs, 11-14
  // converter (Q into tensor memory; quantized cache: K and V too), 15 the
  // P.V MMAs
  static constexpr int kPvWarp = 15;
  static constexpr int kThreads = (kPvWarp + 1) * 32;
  static_assert(kStageOffset % 1024 == 0 && kRawOffset % 1024 == 0, "aligned stages");
  static_assert(kStages <= kMaxStages && kRawStages <= kMaxRawStages, "barrier slots");
  static_assert(kSmemBytes <= 232448, "fits the 227 KB per-block limit");
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;    // S buffers [0, 64) and [64, 128)
constexpr uint32_t kOCol = 128;  // O accumulators [128, 256) and [256, 384)
constexpr uint32_t kQCol = 384;  // two Q buffers [384, 448), [448, 512) (bf16 or f16 pairs)
constexpr float kRescaleLog2 = 8.f;

// bf16 operands (bf16 cache); f16 operands (quantized cache: E4M3 values and
// NVFP4 code x block-scale products are f16 values, and Q is prescaled by a
// power of two into f16's range)
template <bool Q8>
__host__ __device__ constexpr uint32_t idesc_s() {
  return Q8 ? umma::idesc_f16_f32(kRows, kT, false) : umma::idesc_bf16_f32(kRows, kT, false);
}
template <bool Q8>
__host__ __device__ constexpr uint32_t idesc_o() {
  return Q8 ? umma::idesc_f16_f32(kRows, kD, true) : umma::idesc_bf16_f32(kRows, kD, true);
}

__device__ __forceinline__ void tma_box3(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                         int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_box2(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Box {w, 1} at rows r0..r3 of a 2-D map: the four rows of the box (its w
// elements each) back to back from dst (128-byte aligned).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct Maps {
  // bf16: [rows][H_kv][128] elements, box {64, 1, 16}; E4M3: bytes, box
  // {128, 1, 16}; NVFP4 codes: bytes [rows][H_kv][64], box {64, 1, 16}
  CUtensorMap k3, v3;  // (box path)
  // the same as [rows * H_kv][row], box {64 | 128 | 64, 1}
  CUtensorMap k2, v2;  // (gather path)
  // NVFP4 block scales as bytes [rows][H_kv * 8]: box {16, 16} (box path) and
  // {16, 1} (gather path) -- the 8-byte scale rows of heads 2i and 2i + 1
  CUtensorMap ks, vs, ks2, vs2;
};

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t bars;    // shared address of the first mbarrier
  float* merge;     // m, l per O buffer, then the epilogue's merge scratch
  volatile int* abort_flag;
  int32_t* hdr;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) { return c.bars + 8 * i; }

// Bounded wait that also gives up when the abort flag is raised.
__device__ __forceinline__ bool wait_bar(const Ctx& c, int i, uint32_t parity,
                                         unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t bar = bar_addr(c, i);
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*c.abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        set_error(c.hdr, DA_DEVERR_TIMEOUT);
        *c.abort_flag = 1;
        return false;
      }
    }
  }
}

// A unit: KV head h of one (row, split) item.
struct TcUnit {
  int slot, b, h, t_begin, t_end;
  bool single;
};

__device__ __forceinline__ TcUnit tc_unit(const Launch& p, int u) {
  const int4 d = __ldg(reinterpret_cast<const int4*>(p.item_desc) + u / p.H_kv);
  TcUnit x;
  x.single = d.x < 0;
  x.slot = x.single ? ~d.x : d.x;
  x.b = x.slot / p.max_splits;
  x.h = u % p.H_kv;
  x.t_begin = d.y * kT;
  x.t_end = min(d.z * kT, d.w);
  return x;
}

// ---------------------------------------------------------------- producer
// Warps 8 and 9: warp w issues the copies of the tiles g with g % 2 == w
// (and warp 8 each unit's Q rows); both walk every unit and tile.  Box path: a tile's 16-entry group j is copied by one lane; the
// page words of a unit's tiles are loaded eight tiles at a time, a batch
// ahead of the copies that use them (lane l holds the word of group l % 4 of
// tile l / 4 of the batch), and the next unit's descriptor and first batch
// are loaded during the current unit, so the copies never wait on a lookup.
// Gather path: lane j < 16 owns the 4-entry group j of each tile, its words
// loaded one tile ahead.
template <int KT>
__device__ void producer(const Launch& p, const Ctx& c, const Maps& m, int n_units, bool box,
                         int R) {
  constexpr bool Q8 = KT != 0;  // a quantized cache (E4M3 or NVFP4)
  using L = Lay<KT>;
  // the stages this role fills: raw stages of cache bytes, or the operand stages
  constexpr int kNS = Q8 ? L::kRawStages : L::kStages;
  constexpr int kFullB = Q8 ? kRawFull0 : kFull0, kEmptyB = Q8 ? kRawEmpty0 : kEmpty0;
  // quantized cache: warp 8 alone copies (a tile is 8 box copies of codes,
  // plus 8 of NVFP4 scales, not 16 of bf16 halves)
  constexpr int kWarpsCopying = Q8 ? 1 : 2;
  const int lane = threadIdx.x & 31;
  const int pw = (threadIdx.x >> 5) - 8;  // producer warp 0 or 1: tiles of its parity
  if (pw >= kWarpsCopying) return;
  uint32_t g = 0;
  bool bad = false;
  // table word holding entry `tok` (0 past the split or for a contiguous cache)
  auto word_of = [&](const TcUnit& x, int tok) -> int {
    if (tok >= x.t_end || p.layout == DA_KV_CONTIGUOUS) return 0;
    if (p.layout == DA_KV_PAGED) return __ldg(p.table + (size_t)x.b * p.width + tok / p.page_size);
    return __ldg(p.table + (size_t)x.b * p.width + tok);
  };
  // cache row of entry `tok`, or -1 when the entry is past the split or its
  // page / slot is out of range
  auto row_of = [&](const TcUnit& x, int tok, int word) -> long long {
    if (tok >= x.t_end) return -1;
    if (p.layout == DA_KV_CONTIGUOUS) return (long long)x.b * p.width + tok;
    if (word < 0 || word >= p.num_blocks) {
      bad = true;
      return -1;
    }
    if (p.layout == DA_KV_PAGED) return (long long)word * p.page_size + tok % p.page_size;
    return word;
  };
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  // box path: the word of lane l for batch `bt` (tiles 8 bt .. 8 bt + 7) of unit x
  auto batch_word = [&](const TcUnit& x, int bt) -> int {
    return word_of(x, x.t_begin + (8 * bt + (lane >> 2)) * kT + (lane & 3) * 16);
  };
  bool alive = true;
  TcUnit x = tc_unit(p, blockIdx.x);  // blockIdx.x < n_units (the kernel checked)
  int w_first = box ? batch_word(x, 0) : 0;
  for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
    const int u_next = u + (int)gridDim.x;
    const bool has_next = u_next < n_units;
    const TcUnit xn = has_next ? tc_unit(p, u_next) : x;  // in flight during this unit
    const int n_sub = (x.t_end - x.t_begin + kT - 1) / kT;
    int w_cur = w_first, w_nxt = 0, w_n0 = 0;
    if (box && n_sub > 8) w_nxt = batch_word(x, 1);
    // gather path: this lane's four words of the current and the next tile
    int wg[4] = {0, 0, 0, 0}, wg_n[4] = {0, 0, 0, 0};
    if (!box && lane < 16)
      for (int i = 0; i < 4; ++i) wg[i] = word_of(x, x.t_begin + lane * 4 + i);
    const int last_batch = (n_sub - 1) / 8;
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int t0 = x.t_begin + i * kT;
      const int st = g % kNS;
      if (box) {
        if (i > 0 && (i & 7) == 0) {  // next batch: its words were loaded a batch ago
          w_cur = w_nxt;
          if ((i >> 3) + 1 <= last_batch) w_nxt = batch_word(x, (i >> 3) + 1);
        }
        if (i == 8 * last_batch && has_next) w_n0 = batch_word(xn, 0);  // the next unit's
      } else if (lane < 16 && t0 + kT < x.t_end) {
        for (int k = 0; k < 4; ++k) wg_n[k] = word_of(x, t0 + kT + lane * 4 + k);
      }
      if (kWarpsCopying == 2 && (int)(g & 1) != pw) {  // the other producer warp's tile
        if (!box && lane < 16)
          for (int k = 0; k < 4; ++k) wg[k] = wg_n[k];
        continue;
      }
      if (!wait_w(kEmptyB + st, ((g / kNS) & 1) ^ 1)) {
        alive = false;
        break;
      }
      const uint32_t full = bar_addr(c, kFullB + st);
      if (lane == 0) mbar_arrive_expect_tx(full, Q8 ? L::kRawTxBytes : kStageBytes);
      __syncwarp();
      if constexpr (Q8) {
        // E4M3 rows (128 bytes) or NVFP4 code rows (64 bytes) into a raw
        // stage, row-major: K then V; NVFP4 block scales after them (the
        // 16-byte scale rows of heads 2i and 2i + 1, i = h / 2)
        constexpr int kRow = L::kRawCodeBytes / kT;  // code bytes a row
        const uint32_t kdst = c.sbase + L::kRawOffset + st * L::kRawStageBytes;
        const uint32_t vdst = kdst + L::kRawCodeBytes;
        const uint32_t ksdst = kdst + 2 * L::kRawCodeBytes, vsdst = ksdst + L::kRawScaleBytes;
        const int sx = (x.h & ~1) * 8;  // first scale byte of the head pair
        if (box) {
          if ((lane >> 2) == (i & 7)) {
            const int grp = lane & 3;
            long long r = row_of(x, t0 + grp * 16, w_cur);
            if (r < 0) r = 0;
            tma_box3(kdst + grp * 16 * kRow, &m.k3, 0, x.h, (int)r, full);
            tma_box3(vdst + grp * 16 * kRow, &m.v3, 0, x.h, (int)r, full);
            if constexpr (KT == 2) {
              tma_box2(ksdst + grp * 16 * 16, &m.ks, sx, (int)r, full);
              tma_box2(vsdst + grp * 16 * 16, &m.vs, sx, (int)r, full);
            }
          }
        } else if (lane < 16) {
          int rr[4], rs[4];
          for (int k = 0; k < 4; ++k) {
            const long long r = row_of(x, t0 + lane * 4 + k, wg[k]);
            rs[k] = (int)(r < 0 ? 0 : r);
            rr[k] = (int)((r < 0 ? 0 : r) * p.H_kv + x.h);
          }
          tma_gather4(kdst + lane * 4 * kRow, &m.k2, 0, rr[0], rr[1], rr[2], rr[3], full);
          tma_gather4(vdst + lane * 4 * kRow, &m.v2, 0, rr[0], rr[1], rr[2], rr[3], full);
          if constexpr (KT == 2) {
            tma_gather4(ksdst + lane * 128, &m.ks2, sx, rs[0], rs[1], rs[2], rs[3], full);
            tma_gather4(vsdst + lane * 128, &m.vs2, sx, rs[0], rs[1], rs[2], rs[3], full);
          }
          for (int k = 0; k < 4; ++k) wg[k] = wg_n[k];
        }
      } else {
        const uint32_t kdst = c.sbase + L::kStageOffset + st * kStageBytes;
        const uint32_t vdst = kdst + kTileBytes;
        if (box) {
          if ((lane >> 2) == (i & 7)) {
            const int grp = lane & 3;
            long long r = row_of(x, t0 + grp * 16, w_cur);
            if (r < 0) r = 0;
            for (int half = 0; half < 2; ++half) {
              const uint32_t off = half * kRegion + grp * 16 * 128;
              tma_box3(kdst + off, &m.k3, 64 * half, x.h, (int)r, full);
              tma_box3(vdst + off, &m.v3, 64 * half, x.h, (int)r, full);
            }
          }
        } else if (lane < 16) {
          int rr[4];
          for (int k = 0; k < 4; ++k) {
            const long long r = row_of(x, t0 + lane * 4 + k, wg[k]);
            rr[k] = (int)((r < 0 ? 0 : r) * p.H_kv + x.h);
          }
          for (int half = 0; half < 2; ++half) {
            const uint32_t off = half * kRegion + lane * 4 * 128;
            tma_gather4(kdst + off, &m.k2, 64 * half, rr[0], rr[1], rr[2], rr[3], full);
            tma_gather4(vdst + off, &m.v2, 64 * half, rr[0], rr[1], rr[2], rr[3], full);
          }
          for (int k = 0; k < 4; ++k) wg[k] = wg_n[k];
        }
      }
    }
    x = xn;
    w_first = w_n0;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(p.hdr, DA_DEVERR_INDEX);
  // leave no copy in flight into this CTA's shared memory (on the normal path
  // every stage was consumed and these waits return at once).  A warp waits
  // only for its own copies: tiles t < g of its parity (after a time-out, g
  // is the tile it did not copy), which fill the stages of its parity.
  static_assert(kNS % kWarpsCopying == 0, "a stage is filled by one producer warp");
  if (lane == 0) {
    for (int st = pw; st < kNS; st += kWarpsCopying) {
      const int last = (int)g - 1 - (((int)g - 1 - st) % kNS + kNS) % kNS;
      if (last >= 0 && !mbar_wait(bar_addr(c, kFullB + st), (last / kNS) & 1))
        set_error(p.hdr, DA_DEVERR_TIMEOUT);
    }
  }
}

// ---------------------------------------------------------------- converter
// Warps 11-14.  Per unit, once the S MMAs of the unit two back have released
// Q buffer qb (kQFree), each thread writes one MMA row of Q into tensor
// memory -- warp w owns lanes 32 (w % 4) .. + 31 -- as bf16 pairs (bf16
// cache) or as f16 pairs prescaled (quantized cache, q_prescale_exp); rows
// past the group are zeros; then the MMA thread is told (kQConv).  The Q of
// the next unit is written while the current one runs.  Quantized cache
// only: per tile, once its bytes are in raw stage
// g % kRawStages and operand stage g % kStages is free (the PV kStages
// tiles back completed), K and V are written as f16 into the operand stage (NVFP4: each
// code times its block scale, multiplied in f16) in the 128-byte-swizzled
// K-major layout the tensor core reads -- eight lanes per row, so every load
// reads four whole rows, and lanes jj and
// jj + 4 (same chunk pair, other 64-dim region) store their two chunks in
// opposite orders, so the eight lanes of a store phase hit eight different
// bank groups -- and both stages are handed on.
template <int R, int KT>
__device__ void converter(const Launch& p, const Ctx& c, uint32_t tmem, int n_units, bool box) {
  using L = Lay<KT>;
  constexpr bool Q8 = KT != 0;
  constexpr int kGp = kRows / R;  // rows per copy of the group
  const int ct = threadIdx.x - 11 * 32;  // 0..127
  const int warp = threadIdx.x >> 5, lane = ct & 31;
  const int qrow = 32 * (warp & 3) + lane;  // the MMA row (tensor-memory lane) of Q it writes
  const int jq = qrow % kGp;                // that row's head in the group
  const int G = p.H_q / p.H_kv;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  uint32_t g = 0, nq = 0;
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto arrive_w = [&](int bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, bar));
  };
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nq) {
    const TcUnit x = tc_unit(p, u);
    const int n_sub = (x.t_end - x.t_begin + kT - 1) / kT;
    const int qb = nq & 1;
    // ---- Q into tensor-memory columns kQCol + 64 qb .. + 63 (dims 2c, 2c+1 in column c)
    if (!wait_w(kQFree0 + qb, ((nq >> 1) & 1) ^ 1)) return;
    umma::fence_after_sync();
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((size_t)x.b * p.H_q + (size_t)x.h * G + (jq < G ? jq : 0)) * kD);
      float sc = 1.f;
      if constexpr (Q8) {
        float mx = 0.f;
        if (jq < G) {
#pragma unroll 4
          for (int i = 0; i < kD / 8; ++i) mx = fmaxf(mx, bf16x8_absmax(__ldg(src + i)));
        }
        sc = exp2_int(q_prescale_exp(mx));
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 wi = jq < G ? __ldg(src + half * 8 + i) : make_uint4(0, 0, 0, 0);
          const uint32_t v[4] = {wi.x, wi.y, wi.z, wi.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if constexpr (Q8) {
              const __half2 hh = __floats2half2_rn(__uint_as_float(v[e] << 16) * sc,
                                                   __uint_as_float(v[e] & 0xffff0000u) * sc);
              r32[4 * i + e] = *reinterpret_cast<const uint32_t*>(&hh);
            } else {
              r32[4 * i + e] = v[e];  // the bf16 pair as it is
            }
          }
        }
        umma::st_32x32b_x32_u(lane_base + kQCol + qb * 64 + half * 32, r32);
      }
      umma::wait_st();
    }
    umma::fence_before_sync();
    arrive_w(kQConv0 + qb);
    if constexpr (Q8) {  // (bf16: TMA fills the operand stages)
      // ---- K and V of every tile
      const int jj = ct & 7;        // 16-byte piece (dims 16 jj .. 16 jj + 15) of a row
      const int r0 = ct >> 3;       // rows r0, r0 + 16, r0 + 32, r0 + 48 of a tile
      for (int i = 0; i < n_sub; ++i, ++g) {
        const int rs = g % L::kRawStages, os = g % L::kStages;
        if (!wait_w(kRawFull0 + rs, (g / L::kRawStages) & 1)) return;
        if (!wait_w(kEmpty0 + os, ((g / L::kStages) & 1) ^ 1)) return;
        const uint8_t* raw = c.smem + L::kRawOffset + rs * L::kRawStageBytes;
        uint8_t* op = c.smem + L::kStageOffset + os * kStageBytes;
  #pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
  #pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int row = r0 + 16 * q4;
            uint32_t h[8];  // f16 pairs of dims 16 jj .. 16 jj + 15, in order
            if constexpr (KT == 2) {
              // sixteen E2M1 codes and their one E4M3 block scale (byte jj of
              // the head's eight), each exact in f16, multiplied exactly
              const uint2 cw = *reinterpret_cast<const uint2*>(raw + kv * L::kRawCodeBytes +
                                                               row * (kD / 2) + jj * 8);
              const int srow = box ? row * 16 : (row >> 2) * 128 + (row & 3) * 16;
              const uint32_t sb = raw[2 * L::kRawCodeBytes + kv * L::kRawScaleBytes + srow +
                                      (x.h & 1) * 8 + jj];
              const uint32_t s2 = __byte_perm(e4m3x2_to_f16x2(sb), 0, 0x1010);
              uint32_t lo4[4], hi4[4];
              e2m1x8_to_f16x2(cw.x, lo4);
              e2m1x8_to_f16x2(cw.y, hi4);
  #pragma unroll
              for (int e = 0; e < 4; ++e) {
                h[e] = hmul2(lo4[e], s2);
                h[4 + e] = hmul2(hi4[e], s2);
              }
            } else {
              const uint4 b = *reinterpret_cast<const uint4*>(raw + kv * L::kRawCodeBytes +
                                                              row * kD + jj * 16);
              const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
  #pragma unroll
              for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_to_f16x2(wb[e]);
                h[2 * e + 1] = e4m3x2_to_f16x2(wb[e] >> 16);
              }
            }
            // dims 16 jj .. +7 and +8 .. +15: region jj / 4, chunks 2 (jj % 4) and +1
            uint8_t* rbase = op + kv * kTileBytes + (jj >> 2) * kRegion + row * 128;
            const int ch = 2 * (jj & 3);
            const int sw = jj >> 2;  // 0: chunk ch first, 1: chunk ch + 1 first
            const uint4 lo = make_uint4(h[0], h[1], h[2], h[3]);
            const uint4 hi = make_uint4(h[4], h[5], h[6], h[7]);
            *reinterpret_cast<uint4*>(rbase + (((ch + sw) ^ (row & 7)) << 4)) = sw ? hi : lo;
            *reinterpret_cast<uint4*>(rbase + (((ch + 1 - sw) ^ (row & 7)) << 4)) = sw ? lo : hi;
          }
        }
        fence_proxy_async();
        arrive_w(kFull0 + os);
        arrive_w(kRawEmpty0 + rs);
      }
    }
  }
}

// ---------------------------------------------------------------- MMA issue
// Two issuing threads, so that S(g+1) never waits behind PV(g), which needs
// the softmax of tile g: warp 10 issues the S MMAs, warp kPvWarp the P.V
// MMAs.  A tcgen05.commit tracks the MMAs of its own thread, so each thread's
// commits free exactly what its MMAs read.
template <int KT>
__device__ void mma_s(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  constexpr bool Q8 = KT != 0;  // a quantized cache (E4M3 or NVFP4)
  using L = Lay<KT>;
  constexpr int kStages = L::kStages;
  constexpr uint32_t kIdescS = idesc_s<Q8>();
  // K-major tiles, 128-byte swizzle: 8-row groups 1024 bytes apart
  const uint64_t b_k0 =
      umma::smem_desc(c.sbase + L::kStageOffset, 16, 1024, umma::kSwizzle128B);
  uint32_t g = 0, nq = 0;
  // time-out test hook: a wait that runs out, then the abort path
  if (p.test_stall && !wait_bar(c, kStall, 0, kTestStallNs)) return;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nq) {
    const TcUnit x = tc_unit(p, u);
    const int n_sub = (x.t_end - x.t_begin + kT - 1) / kT;
    const int qb = nq & 1;
    if (!wait_bar(c, kQConv0 + qb, (nq >> 1) & 1)) return;  // Q in tensor memory
    fence_proxy_async();
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int st = g % kStages;
      const int sb = g & 1;
      if (!wait_bar(c, kFull0 + st, (g / kStages) & 1)) return;
      fence_proxy_async();
      if (!wait_bar(c, kSFree0 + sb, ((g >> 1) & 1) ^ 1)) return;  // S(g-2) was read
      umma::fence_after_sync();
      const uint64_t b0 = b_k0 + (uint64_t)((st * kStageBytes) >> 4);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {  // dims 16k .. 16k + 15
        const uint32_t off = (k / 4) * kRegion + (k % 4) * 32;
        // A = Q in tensor memory (8 columns per 16 dims)
        umma::mma_bf16_ta(tmem + kSCol + sb * kT, tmem + kQCol + qb * 64 + k * 8,
                          b0 + (uint64_t)(off >> 4), kIdescS, k ? 1u : 0u);
      }
      umma::commit(bar_addr(c, kSFull0 + sb));
      if (i == n_sub - 1) umma::commit(bar_addr(c, kQFree0 + qb));
    }
  }
}

// O += P(g) V(g): P sits over the K tile of stage g % kStages (the softmax
// wrote it once S(g) had read that tile), V after it.
template <int KT>
__device__ void mma_pv(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  constexpr bool Q8 = KT != 0;  // a quantized cache (E4M3 or NVFP4)
  using L = Lay<KT>;
  constexpr int kStages = L::kStages;
  static_assert(kStages <= 7, "the eight P slots cover the softmax's lead");
  constexpr uint32_t kIdescO = idesc_o<Q8>();
  const uint64_t b_k0 =
      umma::smem_desc(c.sbase + L::kStageOffset, 16, 1024, umma::kSwizzle128B);
  // V as an MN-major B operand: 64-dim regions kRegion apart, 8-entry groups
  // 1024 bytes apart
  const uint64_t b_v0 = umma::smem_desc(c.sbase + L::kStageOffset + kTileBytes, kRegion, 1024,
                                        umma::kSwizzle128B);
  uint32_t g = 0, nq = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nq) {
    const TcUnit x = tc_unit(p, u);
    const int n_sub = (x.t_end - x.t_begin + kT - 1) / kT;
    const int ob = nq & 1;
    for (int i = 0; i < n_sub; ++i, ++g) {
      if (!wait_bar(c, kPFull0 + (g & 7), (g >> 3) & 1)) return;
      if (i == 0 && !wait_bar(c, kOFree0 + ob, ((nq >> 1) & 1) ^ 1)) return;
      umma::fence_after_sync();
      const uint32_t st = (g % kStages) * kStageBytes;
      const uint64_t ap = b_k0 + (uint64_t)(st >> 4);
      const uint64_t bv = b_v0 + (uint64_t)(st >> 4);
#pragma unroll
      for (int kk = 0; kk < kT / 16; ++kk)
        umma::mma_bf16(tmem + kOCol + ob * kD, ap + (uint64_t)((kk * 32) >> 4),
                       bv + (uint64_t)((kk * 2048) >> 4), kIdescO, (i == 0 && kk == 0) ? 0u : 1u);
      umma::commit(bar_addr(c, kPVDone0 + (g & 7)));
      umma::commit(bar_addr(c, kEmpty0 + (g % kStages)));
    }
    umma::commit(bar_addr(c, kODone0 + ob));  // the unit's O is complete
  }
}

// ---------------------------------------------------------------- softmax + epilogue
// The group's heads are held R = 128 / Gp times in the MMA rows (Gp = the
// power of two >= G, at least 16): row r is head r % Gp of copy r / Gp.  The
// tensor cores compute every row's scores for the whole tile anyway; copy c
// takes only entries [64c/R, 64(c+1)/R) of each tile (its P row is zero
// elsewhere), so a thread's softmax work per tile is 64/R entries and the
// copies run on all four warps.  Each row keeps its own running reference
// value and sum; at the unit's end the R copies of a head are merged in copy
// order, the combine arithmetic of the split/merge step:
//     M = max_c m_c,  L = sum_c 2^(m_c - M) l_c,  O = sum_c 2^(m_c - M) O_c / L.
// All of it depends only on the unit's own data.
template <int R, int KT>
__device__ void softmax_warps(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  constexpr bool Q8 = KT != 0;  // a quantized cache (E4M3 or NVFP4)
  using L = Lay<KT>;
  constexpr int kGp = kRows / R;              // rows per copy
  constexpr int kCpt = kT / R;                // entries of a tile per copy
  constexpr int kCopiesPerWarp = kGp < 32 ? 32 / kGp : 1;
  constexpr int kWarpCols = kCopiesPerWarp * kCpt;  // columns a warp loads from S
  static_assert(kWarpCols == 16 || kWarpCols == 32 || kWarpCols == 64, "load shapes");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = threadIdx.x;  // TMEM lane
  const int cp = row / kGp, j = row % kGp;
  const int G = p.H_q / p.H_kv;
  const bool live = j < G;  // rows past the group compute but are never written
  const int wcol0 = (warp * 32 / kGp) * kCpt;  // first S column this warp loads
  const int col0 = cp * kCpt;                  // first entry of the tile this row takes
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  float* ml = c.merge;  // [2 buffers][m, l][128]
  uint32_t g = 0, nq = 0;
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto arrive_w = [&](int bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, bar));
  };
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nq) {
    const TcUnit x = tc_unit(p, u);
    const int n_sub = (x.t_end - x.t_begin + kT - 1) / kT;
    const int ob = nq & 1;
    // quantized cache: the row's Q was prescaled by 2^e into f16 (the converter
    // derives e from the same 128 values, see q_prescale_exp), so its scores
    // carry that factor; the row takes it back in its softmax scale
    float row_scale = p.scale_log2;
    if constexpr (Q8) {
      if (live) {
        const uint4* qr = reinterpret_cast<const uint4*>(
            p.q + ((size_t)x.b * p.H_q + (size_t)x.h * G + j) * kD);
        float mx = 0.f;
#pragma unroll 4
        for (int i = 0; i < kD / 8; ++i) mx = fmaxf(mx, bf16x8_absmax(__ldg(qr + i)));
        row_scale *= exp2_int(-q_prescale_exp(mx));
      }
    }
    const uint32_t o_col = kOCol + ob * kD;
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int sb = g & 1;
      if (!wait_w(kSFull0 + sb, (g >> 1) & 1)) return;
      umma::fence_after_sync();
      float s[kCpt];
      {
        float w[kWarpCols];
        const uint32_t a = lane_base + kSCol + sb * kT + wcol0;
        if constexpr (kWarpCols == 16) {
          umma::ld_32x32b_x16(a, w);
        } else if constexpr (kWarpCols == 32) {
          umma::ld_32x32b_x32(a, w);
        } else {
          umma::ld_32x32b_x32(a, *reinterpret_cast<float(*)[32]>(w));
          umma::ld_32x32b_x32(a + 32, *reinterpret_cast<float(*)[32]>(w + 32));
        }
        umma::wait_ld();
        const bool upper = kCopiesPerWarp == 2 && lane >= 16;
#pragma unroll
        for (int k = 0; k < kCpt; ++k) s[k] = upper ? w[kCpt + k] : w[k];
      }
      umma::fence_before_sync();
      arrive_w(kSFree0 + sb);
      const int n_valid = min(kT, x.t_end - (x.t_begin + i * kT)) - col0;
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < kCpt; ++k) {
        // padding rows score 0 everywhere (their Q rows hold arbitrary bytes)
        s[k] = !live ? 0.f : (k < n_valid) ? s[k] * row_scale : -INFINITY;
        mt = fmaxf(mt, s[k]);
      }
      // the reference value moves on the row's first scores and when a score
      // exceeds it by more than 2^8
      const bool move = mt > m_used + kRescaleLog2 || (m_used == -INFINITY && mt > -INFINITY);
      const float m_new = move ? mt : m_used;
      const float alpha = (move && m_used > -INFINITY) ? ex2(m_used - m_new) : 1.f;
      float sum = 0.f;
      uint32_t pk[kCpt / 2];
#pragma unroll
      for (int k = 0; k < kCpt; k += 2) {
        const float p0 = (m_new == -INFINITY) ? 0.f : ex2(s[k] - m_new);
        const float p1 = (m_new == -INFINITY) ? 0.f : ex2(s[k + 1] - m_new);
        sum += p0;
        sum += p1;
        if constexpr (Q8) {  // f16 operands
          const __half2 h = __floats2half2_rn(p0, p1);
          pk[k / 2] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
          const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          pk[k / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      l = fmaf(l, alpha, sum);
      // rescale the row's O when its reference value moved; the previous P.V
      // must have landed first
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!wait_w(kPVDone0 + ((g - 1) & 7), ((g - 1) >> 3) & 1)) return;
        umma::fence_after_sync();
#pragma unroll 1
        for (int ch = 0; ch < kD / 32; ++ch) {
          float o[32];
          umma::ld_32x32b_x32(lane_base + o_col + ch * 32, o);
          umma::wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          umma::st_32x32b_x32(lane_base + o_col + ch * 32, o);
        }
        umma::wait_st();
      }
      m_used = m_new;
      // P row (64 bf16 = 128 bytes: this copy's entries, zeros elsewhere) over
      // the K tile of this tile's stage, in the 128-byte-swizzled K-major
      // layout (S(g), the K tile's only reader, has completed)
      uint8_t* prow = c.smem + L::kStageOffset + (g % L::kStages) * kStageBytes + row * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4 v = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < kCpt / 8; ++q)
          if (cc == col0 / 8 + q) v = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        *reinterpret_cast<uint4*>(prow + ((cc ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async();
      umma::fence_before_sync();
      arrive_w(kPFull0 + (g & 7));
    }
    // hand the rows' (m, l) to the epilogue warps once the epilogue of the
    // unit that used this O buffer before has read its own
    if (!wait_w(kOFree0 + ob, ((nq >> 1) & 1) ^ 1)) return;
    ml[ob * 2 * kRows + row] = m_used;
    ml[ob * 2 * kRows + kRows + row] = l;
    arrive_w(kEpiReady0 + ob);
  }
}

// ---------------------------------------------------------------- epilogue
// Warps 4-7 (warp 4 + q reads TMEM lanes 32q .. 32q + 31, the rows of softmax
// warp q).  Per unit: merge the R copies of each head in copy order,
//     M = max_c m_c,  L = sum_c 2^(m_c - M) l_c,  O = sum_c 2^(m_c - M) O_c,
// and write O / L (bf16 output of a single-split row, else the fp32 partial
// and its LSE in log2 units).  Thread t of the group, for each 32-column
// chunk, sums the R copies of head t % Gp over 32/R of the columns.
template <int R, int KT>
__device__ void epilogue_warps(const Launch& p, const Ctx& c, uint32_t tmem, int n_units) {
  constexpr bool Q8 = KT != 0;  // a quantized cache (E4M3 or NVFP4)
  constexpr int kGp = kRows / R;
  constexpr int kCols = 32 / R;  // columns of a chunk a thread sums
  const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int row = q * 32 + lane;  // TMEM lane = row of the MMA
  const int G = p.H_q / p.H_kv;
  const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
  const float* ml = c.merge;
  float* ob_s = c.merge + 2 * 2 * kRows;  // [128][33]
  const int jt = row % kGp, kq = row / kGp;  // the head and column slice this thread sums
  uint32_t nq = 0;
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nq) {
    const TcUnit x = tc_unit(p, u);
    const int ob = nq & 1;
    // the four warps leave together: one that gave up while another got
    // through would leave the other waiting at the named barrier below
    const bool ok = wait_w(kEpiReady0 + ob, (nq >> 1) & 1) && wait_w(kODone0 + ob, (nq >> 1) & 1);
    if (named_bar_or(1, 128, !ok)) return;
    umma::fence_after_sync();
    const float* m_s = ml + ob * 2 * kRows;
    const float* l_s = m_s + kRows;
    const uint32_t o_col = kOCol + ob * kD;
    // the merged (M, L) of head jt; this row's weight in it
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int cq = 0; cq < R; ++cq) M = fmaxf(M, m_s[cq * kGp + jt]);
#pragma unroll
    for (int cq = 0; cq < R; ++cq) {
      const float mq = m_s[cq * kGp + jt];
      L += (mq == -INFINITY) ? 0.f : ex2(mq - M) * l_s[cq * kGp + jt];
    }
    // this row is copy kq of head jt: its weight in the head's merge
    const float m_row = m_s[row];
    const float f = (m_row == -INFINITY) ? 0.f : ex2(m_row - M);
    const bool writer = jt < G;
    const int hq = x.h * G + jt;
    // (a quantized cache's V scale multiplies the output once, here)
    const float inv = ((L > 0.f) ? 1.f / L : 0.f) * (Q8 ? p.v_scale : 1.f);
#pragma unroll 1
    for (int ch = 0; ch < kD / 32; ++ch) {
      float o[32];
      umma::ld_32x32b_x32(lane_base + o_col + ch * 32, o);
      umma::wait_ld();
      float v[kCols];
      if constexpr (R == 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = o[k];
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) ob_s[row * 33 + k] = o[k] * f;
        named_bar_sync(1, 128);
#pragma unroll
        for (int k = 0; k < kCols; ++k) {
          float a = ob_s[jt * 33 + kq * kCols + k];
#pragma unroll
          for (int cq = 1; cq < R; ++cq) a += ob_s[(cq * kGp + jt) * 33 + kq * kCols + k];
          v[k] = a;
        }
        named_bar_sync(1, 128);
      }
      if (writer) {
        const int d0 = ch * 32 + kq * kCols;
        if (x.single) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + ((size_t)x.b * p.H_q + hq) * kD + d0);
#pragma unroll
          for (int k = 0; k < kCols; k += 2) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[k] * inv, v[k + 1] * inv);
            dst[k / 2] = *reinterpret_cast<const uint32_t*>(&h);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.o_part + ((size_t)x.slot * p.H_q + hq) * kD + d0);
#pragma unroll
          for (int k = 0; k < kCols; k += 4)
            dst[k / 4] = make_float4(v[k] * inv, v[k + 1] * inv, v[k + 2] * inv, v[k + 3] * inv);
        }
      }
    }
    umma::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, kOFree0 + ob));
    if (writer && kq == 0) {
      const float lse2 = (L > 0.f) ? M + lg2(L) : -INFINITY;
      if (x.single)
        p.lse[(size_t)x.b * p.H_q + hq] = (L > 0.f) ? lse2 * kLn2 : -INFINITY;
      else
        p.lse_part[(size_t)x.slot * p.H_q + hq] = lse2;
    }
  }
}

template <int R, int KT>
__global__ void __launch_bounds__(Lay<KT>::kThreads, 1)
    split_gqa_tc_kernel(Launch p, const __grid_constant__ Maps maps, int box) {
  using L = Lay<KT>;
  constexpr bool Q8 = KT != 0;
  constexpr int kThreads = L::kThreads;
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.bars = c.sbase + L::kBarOffset;
  c.merge = reinterpret_cast<float*>(smem + L::kMergeOffset);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortSlot);
  c.hdr = p.hdr;
  const int warp = threadIdx.x >> 5;
  wait_prior_grid();  // the plan kernel's outputs
  allow_next_grid();
  const int n_items = p.hdr[kHdrNWork], n_empty = p.hdr[kHdrNEmpty];
  const int n_units = (n_items - n_empty) * p.H_kv;  // units with tiles, listed first
  const int G = p.H_q / p.H_kv;
  // units of empty rows (listed last): out = 0, lse = -inf
  for (int e = n_units + blockIdx.x; e < n_items * p.H_kv; e += gridDim.x) {
    const TcUnit x = tc_unit(p, e);  // an empty row has one split
    for (int i = threadIdx.x; i < G * kD; i += kThreads)
      p.out[((size_t)x.b * p.H_q + x.h * G) * kD + i] = __float2bfloat16_rn(0.f);
    for (int i = threadIdx.x; i < G; i += kThreads)
      p.lse[(size_t)x.b * p.H_q + x.h * G + i] = -INFINITY;
  }
  if ((int)blockIdx.x >= n_units) return;  // uniform across the CTA
  if (c.sbase & 1023u) {  // the swizzled layouts need 1024-byte-aligned shared memory
    if (threadIdx.x == 0) set_error(p.hdr, DA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;  // tcgen05.commit or the producer's expect_tx arrive
      if ((i >= kSFree0 && i < kSFree0 + 2) || (i >= kPFull0 && i < kPFull0 + 8) ||
          (i >= kEpiReady0 && i < kEpiReady0 + 2) || (i >= kOFree0 && i < kOFree0 + 2))
        count = 4;  // the four softmax (or, for kOFree, epilogue) warps
      if (i == kDrain) count = 2;  // the S and the P.V issuing threads
      // quantized cache: the four converter warps fill the operand stages, free
      // the raw stages and report each converted Q buffer
      if ((Q8 && ((i >= kFull0 && i < kFull0 + kMaxStages) ||
                  (i >= kRawEmpty0 && i < kRawEmpty0 + kMaxRawStages))) ||
          (i >= kQConv0 && i < kQConv0 + 2))
        count = 4;
      mbar_init(bar_addr(c, i), count);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 10) {
    umma::tmem_alloc(c.sbase + L::kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

  if (warp < 4) {
    softmax_warps<R, KT>(p, c, tmem, n_units);
  } else if (warp < 8) {
    epilogue_warps<R, KT>(p, c, tmem, n_units);
  } else if (warp < 10) {
    producer<KT>(p, c, maps, n_units, box != 0, R);
  } else if (warp == 10 || warp == L::kPvWarp) {
    if ((threadIdx.x & 31) == 0) {
      if (warp == 10)
        mma_s<KT>(p, c, tmem, n_units);
      else
        mma_pv<KT>(p, c, tmem, n_units);
      // drain (one commit per issuing thread): its arrival means every MMA
      // this thread issued has completed
      umma::commit(bar_addr(c, kDrain));
    }
  } else {
    converter<R, KT>(p, c, tmem, n_units, box != 0);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 10) {
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

// Stands in for an empty cache in a tensor map (never read by a live entry).
__device__ __nv_bfloat16 g_zero_tile[16 * kD];

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

// A map of `rank` dims (dim 0 = a head row), zero fill past the bounds: bf16
// elements with the 128-byte swizzle (operands copied straight into the
// tensor core's layout), or bytes without swizzle (E4M3 rows, NVFP4 code and
// scale rows, for the converter).
bool encode(CUtensorMap* tm, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, bool bytes) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(tm, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
            const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Copies of the group's rows in the MMA: 128 / (the power of two >= G, >= 16).
int copies_for(int G) {
  int gp = 16;
  while (gp < G) gp <<= 1;
  return kRows / gp;
}

template <int R, int KT>
cudaError_t set_smem() {
  static const cudaError_t e =
      cudaFuncSetAttribute(split_gqa_tc_kernel<R, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay<KT>::kSmemBytes);
  return e;
}

int tc_ctas_per_sm() {
  static const int n = [] {
    if (set_smem<1, 0>() != cudaSuccess) return 1;
    int c = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, split_gqa_tc_kernel<1, 0>,
                                                      Lay<0>::kThreads,
                                                      Lay<0>::kSmemBytes) != cudaSuccess ||
        c < 1)
      c = 1;
    return c;
  }();
  return n;
}
static_assert(Lay<0>::kSmemBytes > 232448 / 2 && Lay<1>::kSmemBytes > 232448 / 2 &&
                  Lay<2>::kSmemBytes > 232448 / 2,
              "every layout runs one CTA per SM (the grid is sized from one)");

template <int R, int KT>
cudaError_t launch_r(const Launch& p, const Maps& m, int box, int grid, cudaStream_t stream) {
  const cudaError_t e = set_smem<R, KT>();
  if (e != cudaSuccess) return e;
  return launch_after(split_gqa_tc_kernel<R, KT>, dim3(grid), dim3(Lay<KT>::kThreads),
                      (size_t)Lay<KT>::kSmemBytes, stream, p, m, box);
}

template <int KT>
cudaError_t launch_q(const Launch& p, const Maps& m, int box, int grid, cudaStream_t stream) {
  switch (copies_for(p.H_q / p.H_kv)) {
    case 8: return launch_r<8, KT>(p, m, box, grid, stream);
    case 4: return launch_r<4, KT>(p, m, box, grid, stream);
    case 2: return launch_r<2, KT>(p, m, box, grid, stream);
    default: return launch_r<1, KT>(p, m, box, grid, stream);
  }
}

}  // namespace

bool gqa_tc_supported(int G, int D) { return G >= 16 && G <= kRows && D == kD; }

int gqa_tc_resident_ctas(int sms) { return tc_ctas_per_sm() * sms; }

cudaError_t launch_split_gqa_tc(const Launch& p, int grid, cudaStream_t stream) {
  const int G = p.H_q / p.H_kv;
  // bf16, E4M3 or NVFP4 caches (kv_type 0, 1, 2; NVFP4 with an even number
  // of KV heads: its scale rows are copied in pairs of heads), one source
  if (!gqa_tc_supported(G, p.D_qk) || p.D_v != kD || p.extra_k || p.kv_type < 0 ||
      p.kv_type > 2 || (p.kv_type == 2 && p.H_kv % 2 != 0))
    return cudaErrorInvalidValue;
  const int kt = p.kv_type;
  const bool q8 = kt != 0;
  const long long rows = (p.layout == DA_KV_CONTIGUOUS) ? (long long)p.B * p.width
                         : (p.layout == DA_KV_PAGED)    ? p.num_blocks * p.page_size
                                                        : p.num_blocks;
  const bool box =
      p.layout == DA_KV_CONTIGUOUS || (p.layout == DA_KV_PAGED && p.page_size % 16 == 0);
  Maps m;
  memset(&m, 0, sizeof m);
  const void* kb = p.k;
  const void* vb = p.v;
  long long r = rows;
  long long heads = p.H_kv;
  if (rows < 1) {  // an empty cache: every entry is masked, copies read zeros
    // (one zero row in the map: every other coordinate lies past its bounds
    // and reads the zero fill)
    void* z = nullptr;
    if (cudaGetSymbolAddress(&z, g_zero_tile) != cudaSuccess) return cudaErrorInvalidValue;
    kb = vb = z;
    r = 1;
    heads = kt == 2 ? 2 : 1;  // NVFP4: 16-byte scale rows
  }
  if (r * heads >= (1ll << 31)) return cudaErrorInvalidValue;  // signed TMA coordinates
  // elements of a head row in the map (NVFP4: its 64 code bytes) and bytes each
  const cuuint64_t row = kt == 2 ? kD / 2 : kD, es = kt == 0 ? 2 : 1;
  const cuuint32_t bx = kt == 0 ? 64u : (cuuint32_t)row;  // box: a 128-byte swizzle span or a row
  const cuuint64_t d3[3] = {row, (cuuint64_t)heads, (cuuint64_t)r};
  const cuuint64_t s3[2] = {row * es, (cuuint64_t)heads * row * es};
  const cuuint32_t b3[3] = {bx, 1, 16};
  const cuuint64_t d2[2] = {row, (cuuint64_t)(r * heads)};
  const cuuint64_t s2[1] = {row * es};
  const cuuint32_t b2[2] = {bx, 1};
  if (!encode(&m.k3, kb, 3, d3, s3, b3, q8) || !encode(&m.v3, vb, 3, d3, s3, b3, q8) ||
      !encode(&m.k2, kb, 2, d2, s2, b2, q8) || !encode(&m.v2, vb, 2, d2, s2, b2, q8))
    return cudaErrorInvalidValue;
  if (kt == 2) {  // block scales [rows][H_kv * 8] bytes, after the codes
    const uint8_t* ks = static_cast<const uint8_t*>(kb) + r * heads * row;
    const uint8_t* vs = static_cast<const uint8_t*>(vb) + r * heads * row;
    const cuuint64_t ds[2] = {(cuuint64_t)heads * 8, (cuuint64_t)r};
    const cuuint64_t ss[1] = {(cuuint64_t)heads * 8};
    const cuuint32_t bs[2] = {16, 16}, bs1[2] = {16, 1};
    if (!encode(&m.ks, ks, 2, ds, ss, bs, true) || !encode(&m.vs, vs, 2, ds, ss, bs, true) ||
        !encode(&m.ks2, ks, 2, ds, ss, bs1, true) || !encode(&m.vs2, vs, 2, ds, ss, bs1, true))
      return cudaErrorInvalidValue;
    return launch_q<2>(p, m, box ? 1 : 0, grid, stream);
  }
  return q8 ? launch_q<1>(p, m, box ? 1 : 0, grid, stream)
            : launch_q<0>(p, m, box ? 1 : 0, grid, stream);
}

}  // namespace da
