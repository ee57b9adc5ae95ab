// Split kernel, tensor-core variant: up to 128 query heads sharing one latent
// KV row of 576 dims whose first 512 dims are the value (MLA-style sparse
// decode, the case "Sparse MLA decode is not batch-invariant" -- FlashMLA
// issue #212 -- reports on).
//
// Both contractions run on tcgen05 tensor cores with fp32 accumulators in
// tensor memory (TMEM):
//     S = Q K^T      M = 128 heads, N = 64 entries, K = 576   (36 MMAs of K=16)
//     O += P V_half  M = 128 heads, N = 256 dims,   K = 64    (4 MMAs)
// O for 128 heads x 512 dims in fp32 would fill all of one SM's tensor memory,
// so a (row, split) item runs as two units, one per half of the value dims;
// each unit computes the full S itself (the same instructions on the same
// data, so both halves see the same bits).
//
// Operand placement.  TMEM columns: Q dims 0..255 [0,128) (the A operand of
// 16 of the 36 S MMAs, so those read only the K tile from shared memory), two
// S buffers [128,192) and [192,256), O [256,512).  Shared memory: Q dims
// 256..575 (80 KB) and two 64-entry KV stages (72 KB each).  P of a tile is
// written into its own KV stage, over the 16 KB of K dims that only S reads
// (dims 256..383 for the low value half, dims 0..127 for the high one), so it
// needs no buffer of its own and is released with the stage.
//
// Pipeline.  S(g) goes into buffer g % 2, so the softmax of tile g-1 can
// overlap the S MMAs of tile g.  S and PV are issued by two threads: PV(g)
// goes out as soon as P(g) is ready and releases its stage, so the copy of
// tile g+2 starts without waiting for S(g+1) to be issued (with two stages,
// the copy latency is otherwise exposed on every tile).
// The softmax touches O only to rescale it (when its running max moves by
// more than 2^8), after the PV before it has landed.  The producer prefetches
// the next tile's rows into L2 while the current stage is in use.
//
// Roles inside a CTA (320 threads; 448 with the E4M3 converter):
//   warps 0-3  softmax: thread i owns head i = TMEM lane i.  It loads its row
//              of Q dims 0..255 into TMEM at the start of a unit, reads its
//              row of S, keeps the running max and sum in fp32, writes P
//              (bf16) into the stage and writes its row of the result.
//   warps 4-7  producer: looks up each entry's cache row and copies the
//              1152-byte latent rows with 16-byte cp.async runs into the
//              128-byte-swizzled K-major layout the tensor core reads; the
//              unit's Q dims 256..575 come by TMA tile copies, issued after
//              the unit's first tile (whose index words were loaded during
//              the previous unit) and once the previous unit's S is done.
//   warp 8     S MMA issue (one thread) and TMEM allocation.
//   warp 9     P.V MMA issue (one thread).
//   warps 10-13  E4M3 cache only: the converter (below).
//
// E4M3 latent cache (one byte per element, one fp32 scale for the scores
// and one for the values).  Every E4M3 value is an f16 value, so the MMAs
// run on f16 operands.  Q: dims 256..575 arrive by TMA as for bf16 and the
// softmax warps rescale them in place, dims 0..255 go to TMEM as f16 -- the
// row times 2^e, e from its largest magnitude, so it lies in f16's range.
// K: the four producer warps copy each row's 576 bytes with 16-byte cp.async
// (consecutive threads take consecutive runs of a row, so a row's copies
// coalesce) into the upper half of the operand stage as three 192-byte
// pieces, piece c of rows 0..63 back to back at 36 KB + 12 KB c; each thread
// arrives on the stage's barrier once its copies have landed.  (Gathers
// through the TMA unit of rows at random addresses proved to be bound by the
// unit's per-request cost, not by HBM.)  The converter warps widen the bytes
// in place into the 128-byte-swizzled f16 layout.  Piece 0 becomes f16 regions
// 0..2, below the raw bytes; pieces 1 and 2 are read into registers and the
// four warps meet at a barrier before regions 3..8 (which cover the raw
// bytes) are written.
// Every wait on an mbarrier is bounded; on time-out the kernel records
// DA_DEVERR_TIMEOUT, every role leaves its loop, outstanding tensor-core work
// is drained (bounded) and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace da {
namespace {

constexpr int kHeads = 128;       // MMA M (query heads, zero-padded)
constexpr int kDqk = 576;
constexpr int kDvHalf = 256;      // value dims per unit
constexpr int kSub = 64;          // entries per sub-tile (MMA N of S, K of P.V)
constexpr int kRegions = kDqk / 64;  // 64-dim swizzle regions of a row
constexpr int kQT = 256;          // dims of Q held in TMEM (A operand)
constexpr int kQTCols = kQT / 2;  // 128 TMEM columns (two bf16 per column)
constexpr int kQSRegions = (kDqk - kQT) / 64;  // 5 smem regions of Q (dims 256..575)
constexpr int kStages = 2;

// shared memory map (bytes)
constexpr int kQSBytes = kQSRegions * kHeads * 128;        // 81920
constexpr int kStageRegion = kSub * 128;                    // 8192
constexpr int kStageBytes = kRegions * kStageRegion;        // 73728
constexpr int kStageOffset = kQSBytes;
constexpr int kPBytes = kHeads * kSub * 2;                  // 16384 (128-byte swizzle)
constexpr int kBarOffset = kStageOffset + kStages * kStageBytes;  // 229376
// Barriers that are signalled once per tile come in pairs indexed by the
// tile's parity.  A parity wait is only unambiguous while the barrier is at
// most one phase behind the phase waited for; the softmax waits for PV
// completion only when it rescales O (and at the epilogue), so a single
// PV-done barrier could be two phases behind there.
enum { kFull0 = 0, kEmpty0 = kFull0 + kStages, kSFull0 = kEmpty0 + kStages,
       kSFree0 = kSFull0 + 2, kPFull0 = kSFree0 + 2, kODone0 = kPFull0 + 2,
       kOFree = kODone0 + 2, kQFull, kQTFull, kQFree, kDrain,
       kStall,  // never signalled: the time-out test hook waits on it
       kRawFull0,  // E4M3 cache: a stage's raw bytes landed (kFull: converted)
       kNumBars = kRawFull0 + kStages };
constexpr int kTmemSlot = kBarOffset + kNumBars * 8;
static_assert(kStageOffset % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle atoms 1024-aligned");
constexpr int kAbortSlot = kTmemSlot + 4;
// the global address of each entry's cache row, two tiles' worth
// (producer lanes -> all producer threads)
constexpr int kRowsSlot = (kAbortSlot + 12 + 15) / 16 * 16;
constexpr int kSmemBytes = kRowsSlot + 2 * 64 * 8;
static_assert(kSmemBytes <= 232448, "fits the 227 KB per-block limit");

// P of a tile sits in its stage over K dims that only S reads: regions 4-5
// (dims 256..383) when the unit takes value dims 0..255, regions 0-1 when it
// takes 256..511.
__host__ __device__ constexpr int p_offset_in_stage(int half) {
  return (half == 0 ? 4 : 0) * kStageRegion;
}
static_assert(2 * kStageRegion == kPBytes, "P fills two regions");

// E4M3 cache: the raw bytes of a tile in the upper half of its stage, as
// three pieces of 192 bytes per row (dims 192 c .. 192 c + 191), piece c of
// the 64 rows back to back
constexpr int kRawInStage = kStageBytes / 2;  // 36864
constexpr int kRawPiece = 192;                // bytes of a row per copy
constexpr int kRawPieces = kDqk / kRawPiece;  // 3
constexpr int kRawPieceBytes = kSub * kRawPiece;  // 12288
static_assert(kRawInStage + kRawPieces * kRawPieceBytes == kStageBytes,
              "raw bytes fill the upper half");
static_assert((kRawPiece / 64) * kStageRegion <= kRawInStage,
              "piece 0's f16 regions end below the raw bytes");
constexpr int kConvBar = 1;                   // named barrier of the converter warps
constexpr int kProdBar = 2;                   // named barrier of the producer warps

// KT: 0 bf16 cache, 1 E4M3 cache (four more warps: the converter)
template <int KT>
constexpr int threads_for() { return KT ? 448 : 320; }
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = kQTCols;  // S buffers at [128, 192) and [192, 256)
constexpr int kKSteps = kDqk / 16;   // 36 MMAs of K = 16 per S tile
constexpr int kEntPerWarp = kSub / 4;  // entries each producer warp gathers
constexpr uint32_t kOCol = 256;      // O accumulator columns [256, 512)
static_assert(kSCol + 2 * kSub == kOCol && kOCol + kDvHalf == kTmemCols, "TMEM budget");
constexpr float kRescaleLog2 = 8.f;

// bf16 operands (bf16 cache) or f16 operands (E4M3 cache)
template <int KT>
constexpr uint32_t idesc_s() {
  return KT ? umma::idesc_f16_f32(kHeads, kSub, false) : umma::idesc_bf16_f32(kHeads, kSub, false);
}
template <int KT>
constexpr uint32_t idesc_o() {
  return KT ? umma::idesc_f16_f32(kHeads, kDvHalf, true)
            : umma::idesc_bf16_f32(kHeads, kDvHalf, true);
}

// TMA copies from a 2-D tensor map (dim 0 = the 576 dims of a row, dim 1 =
// rows) into this CTA's own shared memory, 128-byte swizzle applied by the
// copy engine from the shared-memory address; each completes its bytes on the
// mbarrier at shared address `bar`.

// One box of the map (its box dims) at (col, row).
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* tm, int col, int row,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(row), "r"(bar)
      : "memory");
}

// 32 bytes from global memory (read-only path) as two 16-byte halves; the
// address is 32-byte aligned.
__device__ __forceinline__ void ldg_v8(const void* src, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(src));
}

// Start pulling `bytes` (a multiple of 16) at a 16-byte-aligned address into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;  // shared address of smem[0]
  volatile int* abort_flag;
  int32_t* hdr;
  const CUtensorMap* tm_q;  // q as [B * H_q, 576], box {64, 16}
};

// Rows of a 16-row box of Q a unit loads (heads rounded up to 16).
constexpr int kQBoxRows = 16;

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) {
  return c.sbase + kBarOffset + 8 * i;
}

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

// The units a CTA takes.  Unit 2i + h is value half h of work item i; CTA
// pair q (CTAs 2q, 2q + 1) takes item k * pairs + q in even rounds k and
// k * pairs + (pairs - 1 - q) in odd ones.  The list is sorted largest
// first, so this serpentine deal evens out the pairs' sums, and the two
// halves of an item run at the same time on neighbouring CTAs (all CTAs are
// resident), so the second read of each latent row is served by L2.
// Placement only: no unit's arithmetic depends on its CTA.
__device__ __forceinline__ int next_unit(int u) {
  const int pairs = gridDim.x >> 1, q = blockIdx.x >> 1;
  const int k = (u >> 1) / pairs + 1;
  return 2 * (k * pairs + ((k & 1) ? pairs - 1 - q : q)) + (u & 1);
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

// Latent-cache row holding entry `tok` of row b (H_kv = 1), in two steps so
// that the index load can be in flight while other work is issued:
// latent_fetch loads the table word the entry needs (its page id or slot;
// nothing for a contiguous cache), latent_decode turns it into the row and
// the source (1 for entries from l_main on, which come from the second
// source) and says whether the index is in range.
__device__ __forceinline__ int latent_fetch(const Launch& p, int b, int tok, int l_main) {
  if (tok >= l_main) return __ldg(p.extra_table + (size_t)b * p.extra_width + (tok - l_main));
  if (p.layout == DA_KV_CONTIGUOUS) return 0;
  if (p.layout == DA_KV_PAGED) return __ldg(p.table + (size_t)b * p.width + tok / p.page_size);
  return __ldg(p.table + (size_t)b * p.width + tok);
}

__device__ __forceinline__ bool latent_decode(const Launch& p, int b, int tok, int l_main,
                                              int word, long long* row, int* src) {
  *src = 0;
  if (tok >= l_main) {
    *row = word;
    *src = 1;
    return word >= 0 && word < p.extra_num_blocks;
  }
  if (p.layout == DA_KV_CONTIGUOUS) {
    *row = (long long)b * p.width + tok;
    return true;
  }
  if (p.layout == DA_KV_PAGED) {
    *row = (long long)word * p.page_size + tok % p.page_size;
    return word >= 0 && word < p.num_blocks;
  }
  *row = word;
  return word >= 0 && word < p.num_blocks;
}

// Stands in for an empty cache: dummy copies of masked entries read it.
__device__ __align__(16) __nv_bfloat16 g_zero_row[kDqk];

// ---------------------------------------------------------------- producer
// The four warps copy a tile with 16-byte cp.async, consecutive threads
// taking consecutive 16-byte runs of a row (so a row's copies coalesce); each
// thread arrives on the stage's barrier once its own copies have landed.
// (TMA gathers of rows at random addresses proved bound by the copy unit's
// per-request cost, not by HBM.)  The warps meet at a named barrier per tile
// (the entries' row addresses pass through shared memory), so every wait is
// decided together -- a bounded wait that ran out in one warp ends all four
// -- and none is ever left at the barrier.
template <int KT>
__device__ void producer(const Launch& p, const Ctx& c, int n_units) {
  constexpr int kRowBytes = KT ? kDqk : 2 * kDqk;  // bytes of a cache row
  constexpr int kRunsPerRow = kRowBytes / 16;      // 16-byte runs of a row
  constexpr int kRunsPerThread = kSub * kRunsPerRow / 128;
  static_assert(kSub * kRunsPerRow % 128 == 0, "a tile's runs split evenly over 128 threads");
  const int pt = threadIdx.x - 128;  // 0..127
  const int pw = pt >> 5, pl = pt & 31;
  uint32_t g = 0, n_ne = 0;
  bool alive = true;
  bool bad = false;
  // warp-uniform bounded wait (lane 0 waits, everyone follows its verdict)
  auto wait_w = [&](int bar, uint32_t parity) -> bool {
    int ok = 1;
    if (pl == 0) ok = wait_bar(c, bar, parity) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return !named_bar_or(kProdBar, 128, ok == 0);
  };
  // the main cache (or the zero row standing in for an empty one) and the
  // second source
  const uint8_t* kmain = p.kv_rows < 1 ? reinterpret_cast<const uint8_t*>(g_zero_row)
                                       : reinterpret_cast<const uint8_t*>(p.k);
  const uint8_t* kextra = reinterpret_cast<const uint8_t*>(p.extra_k);
  const int q_boxes = (min(p.H_q, kHeads) + kQBoxRows - 1) / kQBoxRows;  // per region
  // Lane e < 16 of producer warp pw handles entry 16*pw + e of a tile.
  // Table words are loaded two tiles ahead and decoded one tile ahead (the
  // decoded rows of the next tile are prefetched into L2), so the index
  // load's latency stays off the copy path; a unit's first two tiles' words
  // are loaded during the previous unit's last tile.
  // src: 0 = main cache, 1 = second source.  Masked entries (past the end
  // of the split) and bad indices read row 0 of the main cache, so every
  // stage byte holds real data; masked scores are dropped by the softmax.
  const int e_lane = kEntPerWarp * pw + pl;
  auto fetch = [&](const MlaUnit& xu, int t0) -> int {
    const int tok = t0 + e_lane;
    return (pl < kEntPerWarp && tok < xu.t_end) ? latent_fetch(p, xu.b, tok, xu.l_main) : 0;
  };
  auto decode = [&](const MlaUnit& xu, int t0, int word, int& row, int& src, bool& live) {
    row = 0;
    src = 0;
    live = false;
    const int tok = t0 + e_lane;
    if (pl < kEntPerWarp && tok < xu.t_end) {
      long long r;
      int sr;
      const bool good = latent_decode(p, xu.b, tok, xu.l_main, word, &r, &sr);
      bad |= !good;
      if (good) {
        row = (int)r;
        src = sr;
        live = true;
      }
    }
  };
  // the next unit with tiles at or after u
  auto next_live = [&](int u) -> int {
    while (u < n_units && mla_unit(p, u).empty) u = next_unit(u);
    return u;
  };
  uint32_t nq_issued = 0;  // units whose Q copy was issued
  int u = next_live(blockIdx.x);
  MlaUnit x = mla_unit(p, u < n_units ? u : 0);
  int pre_w0 = 0, pre_w1 = 0;  // the unit's first two tiles' words
  if (u < n_units) {
    pre_w0 = fetch(x, x.t_begin);
    pre_w1 = (x.t_begin + kSub < x.t_end) ? fetch(x, x.t_begin + kSub) : 0;
  }
  while (u < n_units && alive) {
    const int un = next_live(next_unit(u));
    const bool has_next = un < n_units;
    const MlaUnit xn = has_next ? mla_unit(p, un) : x;
    // warm L2 with the next unit's query rows (its softmax warps load them
    // into tensor memory at its start)
    if (has_next) {
      const char* qn = reinterpret_cast<const char*>(p.q + (size_t)xn.b * p.H_q * kDqk);
      const int lines = min(p.H_q, kHeads) * kDqk * 2 / 128;
      for (int i = pt; i < lines; i += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + (size_t)i * 128));
    }
    int my_row, my_src, nx_row = 0, nx_src = 0;
    bool my_live, nx_live = false;
    int nx_word = pre_w1;
    decode(x, x.t_begin, pre_w0, my_row, my_src, my_live);
    bool pre_fetched = false;  // the next unit's first words are loaded
    for (int t0 = x.t_begin; t0 < x.t_end; t0 += kSub, ++g) {
      const int stage = g % kStages;
      if (!wait_w(kEmpty0 + stage, ((g / kStages) & 1) ^ 1)) {
        alive = false;
        break;
      }
      // (E4M3 cache: the raw bytes' own barrier; the converter signals kFull)
      const uint32_t full = bar_addr(c, (KT ? kRawFull0 : kFull0) + stage);
      // the row addresses of the tile's entries into shared memory, then run
      // k of the tile (row k / kRunsPerRow, bytes 16 (k % kRunsPerRow) ..)
      // by thread k % 128
      const uint8_t** rows_s = reinterpret_cast<const uint8_t**>(c.smem + kRowsSlot) + (g & 1) * kSub;
      if (pl < kEntPerWarp)
        rows_s[kEntPerWarp * pw + pl] = (my_src ? kextra : kmain) + (size_t)my_row * kRowBytes;
      named_bar_sync(kProdBar, 128);
      const uint32_t st = c.sbase + kStageOffset + stage * kStageBytes;
#pragma unroll 6
      for (int i = 0; i < kRunsPerThread; ++i) {
        const int k = pt + 128 * i;
        const int rr = k / kRunsPerRow, q = k % kRunsPerRow;
        // E4M3: raw piece q / 12, rows back to back; bf16: 64-dim region
        // q / 8, chunk q % 8 of the row, 128-byte swizzle
        const uint32_t dst =
            KT ? st + kRawInStage + (q / 12) * kRawPieceBytes + rr * kRawPiece + (q % 12) * 16
               : st + (q >> 3) * kStageRegion + rr * 128 + (((q & 7) ^ (rr & 7)) << 4);
        cp_async16(dst, rows_s[rr] + q * 16);
      }
      cp_async_mbar_arrive(full);
      // Q dims 256..575 of row b into shared memory once the previous
      // unit's S MMAs are done (after this unit's first tile is on its way):
      // q_boxes 16-row boxes per 64-dim region, spread over the four warps
      // (rows past H_q belong to other rows or read as zeros; those heads'
      // results are never written).  E4M3 cache: the softmax warps then
      // rescale them into f16 in place.
      if (t0 == x.t_begin) {
        if (!wait_w(kQFree, (n_ne & 1) ^ 1)) {
          alive = false;
          break;
        }
        if (pt == 0)
          mbar_arrive_expect_tx(bar_addr(c, kQFull), kQSRegions * q_boxes * kQBoxRows * 128);
        __syncwarp();
        for (int i = pt; i < kQSRegions * q_boxes; i += 128) {
          const int j = i / q_boxes, rb = i % q_boxes;
          tma_tile(c.sbase + j * (kHeads * 128) + rb * (kQBoxRows * 128), c.tm_q, kQT + 64 * j,
                   x.b * p.H_q + rb * kQBoxRows, bar_addr(c, kQFull));
        }
        ++nq_issued;
      }
      // decode the next tile's words (loaded an iteration ago), load the
      // words of the tile after it, and start the next tile's rows towards L2
      if (t0 + kSub < x.t_end) decode(x, t0 + kSub, nx_word, nx_row, nx_src, nx_live);
      if (t0 + 2 * kSub < x.t_end) nx_word = fetch(x, t0 + 2 * kSub);
      // the next unit: its first two tiles' words during this unit's
      // second-to-last tile (or its only one), its first tile's rows towards
      // L2 during the last
      if (has_next && t0 + kSub >= x.t_end && pre_fetched) {
        int r0, s0;
        bool l0;
        decode(xn, xn.t_begin, pre_w0, r0, s0, l0);
        if (l0)
          prefetch_l2(reinterpret_cast<const uint8_t*>(s0 ? p.extra_k : p.k) +
                          (size_t)r0 * kRowBytes,
                      kRowBytes);
      }
      if (has_next && t0 + 2 * kSub >= x.t_end && !pre_fetched) {
        pre_w0 = fetch(xn, xn.t_begin);
        pre_w1 = (xn.t_begin + kSub < xn.t_end) ? fetch(xn, xn.t_begin + kSub) : 0;
        pre_fetched = true;
      }
      if (nx_live && t0 + kSub < x.t_end)
        prefetch_l2(reinterpret_cast<const uint8_t*>(nx_src ? p.extra_k : p.k) +
                        (size_t)nx_row * kRowBytes,
                    kRowBytes);
      my_row = nx_row;
      my_src = nx_src;
      my_live = nx_live;
    }
    if (!alive) break;
    ++n_ne;
    u = un;
    x = xn;
  }
  if (bad) set_error(p.hdr, DA_DEVERR_INDEX);
  // leave no copy in flight into this CTA's shared memory (on the normal path
  // every stage was consumed and these waits return at once)
  cp_async_wait_all();
  if (pt == 0 && nq_issued > 0 && !mbar_wait(bar_addr(c, kQFull), (nq_issued - 1) & 1))
    set_error(p.hdr, DA_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------- MMA issue
// Two issuing threads: warp 8 issues the S MMAs, warp 9 the P.V MMAs, so
// S(g+1) never waits behind P.V(g), which needs the softmax of tile g, and
// P.V(g) goes out as soon as P(g) is ready.  A tcgen05.commit tracks the MMAs
// of its own thread, so each thread's commits free exactly what its MMAs
// read.  The softmax can lead the P.V thread by at most one tile (S(g) needs
// stage g's copy, which needs P.V(g - 2) done), so the per-parity P-ready and
// P.V-done barriers stay within one phase of every wait.
template <int KT>
__device__ void mma_s(const Launch& p, const Ctx& c, uint32_t tmem, int n_units, uint32_t& n_ne) {
  constexpr uint32_t kIdescS = idesc_s<KT>();
  // base descriptors; per-MMA ones differ only by a constant start offset
  const uint64_t b_stage0 =  // K tile, K-major, 128-byte swizzle
      umma::smem_desc(c.sbase + kStageOffset, 16, 1024, umma::kSwizzle128B);
  const uint64_t a_q0 =      // Q dims 256..575, K-major, 128-byte swizzle
      umma::smem_desc(c.sbase, 16, 1024, umma::kSwizzle128B);
  uint32_t g = 0;
  // time-out test hook: a wait that runs out, then the abort path
  if (p.test_stall && !wait_bar(c, kStall, 0, kTestStallNs)) return;
  for (int u = blockIdx.x; u < n_units; u = next_unit(u)) {
    const MlaUnit x = mla_unit(p, u);
    if (x.empty) continue;
    const int n_sub = (x.t_end - x.t_begin + kSub - 1) / kSub;
    if (KT == 0) {  // Q dims 256.. in shared memory (E4M3 cache: rescaled, with kQTFull)
      if (!wait_bar(c, kQFull, n_ne & 1)) return;
      fence_proxy_async();
    }
    if (!wait_bar(c, kQTFull, n_ne & 1)) return;  // Q dims 0..255 in TMEM
    umma::fence_after_sync();
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int stage = g % kStages;
      const int sb = g & 1;
      if (!wait_bar(c, kFull0 + stage, (g / kStages) & 1)) return;
      fence_proxy_async();
      if (!wait_bar(c, kSFree0 + sb, ((g >> 1) & 1) ^ 1)) return;  // S(g-2) was read
      umma::fence_after_sync();
      // S = Q K^T: 36 MMAs of M = 128, N = 64, K = 16 into S buffer sb
      const uint64_t b0 = b_stage0 + (uint64_t)((stage * kStageBytes) >> 4);
      const uint32_t d_s = tmem + kSCol + sb * kSub;
#pragma unroll
      for (int k = 0; k < kKSteps; ++k) {  // K step k: dims 16k .. 16k+15
        const uint64_t b = b0 + (uint64_t)(((k / 4) * kStageRegion + (k % 4) * 32) >> 4);
        if (k < kQT / 16)  // A = Q rows in TMEM (8 columns per 16 dims)
          umma::mma_bf16_ta(d_s, tmem + k * 8, b, kIdescS, k ? 1u : 0u);
        else               // A = Q dims 256.. in shared memory
          umma::mma_bf16(d_s, a_q0 + (uint64_t)((((k - kQT / 16) / 4) * kHeads * 128 +
                                                   (k % 4) * 32) >> 4),
                         b, kIdescS, 1u);
      }
      umma::commit(bar_addr(c, kSFull0 + sb));
      if (i == n_sub - 1) umma::commit(bar_addr(c, kQFree));
    }
    ++n_ne;
  }
}

// O += P(g) V(g): P and V both sit in the stage of tile g.
template <int KT>
__device__ void mma_pv(const Launch& p, const Ctx& c, uint32_t tmem, int n_units, uint32_t& g) {
  constexpr uint32_t kIdescO = idesc_o<KT>();
  const uint64_t b_stage0 =
      umma::smem_desc(c.sbase + kStageOffset, 16, 1024, umma::kSwizzle128B);
  const uint64_t b_v0 =      // V = leading dims of the K tile, MN-major
      umma::smem_desc(c.sbase + kStageOffset, kStageRegion, 1024, umma::kSwizzle128B);
  uint32_t n_ne = 0;
  for (int u = blockIdx.x; u < n_units; u = next_unit(u)) {
    const MlaUnit x = mla_unit(p, u);
    if (x.empty) continue;
    const int n_sub = (x.t_end - x.t_begin + kSub - 1) / kSub;
    for (int i = 0; i < n_sub; ++i, ++g) {
      if (!wait_bar(c, kPFull0 + (g & 1), (g >> 1) & 1)) return;
      if (i == 0 && !wait_bar(c, kOFree, (n_ne & 1) ^ 1)) return;
      umma::fence_after_sync();
      const uint32_t st = (g % kStages) * kStageBytes;
      const uint64_t ap = b_stage0 + (uint64_t)((st + p_offset_in_stage(x.half)) >> 4);
      const uint64_t bv = b_v0 + (uint64_t)((st + 4 * x.half * kStageRegion) >> 4);
#pragma unroll
      for (int kk = 0; kk < kSub / 16; ++kk)
        umma::mma_bf16(tmem + kOCol, ap + (uint64_t)((kk * 32) >> 4),
                       bv + (uint64_t)((kk * 2048) >> 4), kIdescO, (i == 0 && kk == 0) ? 0u : 1u);
      umma::commit(bar_addr(c, kODone0 + (g & 1)));
      umma::commit(bar_addr(c, kEmpty0 + (g % kStages)));
    }
    ++n_ne;
  }
}

// ---------------------------------------------------------------- softmax + epilogue
// bf16 pair (low half = lower dim) times 2^e as an f16 pair (exact but for
// f16 subnormals, see q_prescale_exp).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t v, float sc) {
  const __half2 h = __floats2half2_rn(__uint_as_float(v << 16) * sc,
                                      __uint_as_float(v & 0xffff0000u) * sc);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int KT>
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
  // Q dims 0..255 of head `row` of row b into TMEM columns [0, 128): two bf16
  // per column, the lower dim in the low half; then signal the MMA thread.
  // E4M3 cache: the row times 2^e as f16 (e from the row's largest
  // magnitude, q_prescale_exp) -- dims 0..255 into TMEM the same way, dims
  // 256..575 rescaled in place in the shared-memory Q regions once their TMA
  // copy (kQFull, phase parity `qpar`) has landed; `e` gets the exponent (0
  // for a bf16 cache).  False when a bounded wait ran out.
  // 32-byte loads when q allows them (a row's 1152 bytes keep the alignment):
  // each load instruction touches as many rows as a 16-byte one, for twice
  // the bytes
  const bool q32 = (reinterpret_cast<uintptr_t>(p.q) & 31) == 0;
  auto load_q = [&](int b, uint32_t qpar, int& e) -> bool {
    const bool ok = row < p.H_q;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.H_q + row) * kDqk);
    // dims 128 half .. 128 half + 127 of the row (zeros past the heads)
    auto load_half = [&](int half, uint4 (&w)[16]) {
      if (!ok) {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = make_uint4(0, 0, 0, 0);
      } else if (q32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ldg_v8(qrow + half * 16 + 2 * i, w[2 * i], w[2 * i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = __ldg(qrow + half * 16 + i);
      }
    };
    e = 0;
    if constexpr (KT == 1) {
      // (the loops stay rolled: this runs once per unit, and its code is
      // fetched cold each time)
      uint8_t* qs = c.smem + row * 128;  // + region j * kHeads * 128 + swizzled chunk
      uint32_t mb = 0;                   // magnitude bits, see bf16x8_absmax_bits
      // dims 0..255: into TMEM as bf16 pairs (as for a bf16 cache) while
      // taking the maximum (the TMA copy of dims 256..575 lands meanwhile);
      // rescaled there below
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint4 w[16];
        load_half(half, w);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t r32[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = w[ch * 8 + i];
            mb = bf16x8_absmax_bits(mb, v);
            r32[4 * i + 0] = v.x;
            r32[4 * i + 1] = v.y;
            r32[4 * i + 2] = v.z;
            r32[4 * i + 3] = v.w;
          }
          umma::st_32x32b_x32_u(lane_base + (half * 2 + ch) * 32, r32);
        }
      }
      if (!wait_w(kQFull, qpar)) return false;  // dims 256..575 in shared memory
#pragma unroll 1
      for (int j = 0; j < kQSRegions; ++j)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          mb = bf16x8_absmax_bits(mb, *reinterpret_cast<const uint4*>(
                                          qs + j * (kHeads * 128) + ((cc ^ (row & 7)) << 4)));
      e = q_prescale_exp(bf16_absmax_value(mb));
      const float sc = exp2_int(e);
      umma::wait_st();
#pragma unroll 1
      for (int ch = 0; ch < kQTCols / 32; ++ch) {
        float f[32];
        umma::ld_32x32b_x32(lane_base + ch * 32, f);
        umma::wait_ld();
        uint32_t r32[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r32[i] = bf16x2_to_f16x2_scaled(__float_as_uint(f[i]), sc);
        umma::st_32x32b_x32_u(lane_base + ch * 32, r32);
      }
#pragma unroll 1
      for (int j = 0; j < kQSRegions; ++j)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {  // 8 dims (16 bytes) per chunk, own row only
          uint4* q16 = reinterpret_cast<uint4*>(qs + j * (kHeads * 128) + ((cc ^ (row & 7)) << 4));
          const uint4 v = *q16;
          *q16 = make_uint4(bf16x2_to_f16x2_scaled(v.x, sc), bf16x2_to_f16x2_scaled(v.y, sc),
                            bf16x2_to_f16x2_scaled(v.z, sc), bf16x2_to_f16x2_scaled(v.w, sc));
        }
      fence_proxy_async();  // the S MMAs read these rows
      umma::wait_st();
      umma::fence_before_sync();
      arrive_w(kQTFull);
      return true;
    } else {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint4 w[16];
        load_half(half, w);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t r32[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            r32[4 * i + 0] = w[ch * 8 + i].x;
            r32[4 * i + 1] = w[ch * 8 + i].y;
            r32[4 * i + 2] = w[ch * 8 + i].z;
            r32[4 * i + 3] = w[ch * 8 + i].w;
          }
          umma::st_32x32b_x32_u(lane_base + (half * 2 + ch) * 32, r32);
        }
      }
      umma::wait_st();
      umma::fence_before_sync();
      arrive_w(kQTFull);
      return true;
    }
  };
  bool q_ready = false;  // Q of the coming unit already in TMEM
  int e_next = 0;        // its prescale exponent (E4M3 cache)
  for (int u = blockIdx.x; u < n_units; u = next_unit(u)) {
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
    int e_q = e_next;
    if (!q_ready) {
      // (first unit only: later units get their Q while the previous unit's
      // epilogue is still ahead, see below)
      if (!wait_w(kQFree, (n_ne & 1) ^ 1)) return;
      umma::fence_after_sync();
      if (!load_q(x.b, n_ne & 1, e_q)) return;
    }
    q_ready = false;
    // E4M3 cache: the scores carry Q's factor 2^e; the row takes it back here
    const float row_scale = KT ? p.scale_log2 * exp2_int(-e_q) : p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int sb = g & 1;
      if (!wait_w(kSFull0 + sb, (g >> 1) & 1)) return;
      umma::fence_after_sync();
      float s[64];
      {
        float s_hi[32];
        umma::ld_32x32b_x32(lane_base + kSCol + sb * kSub, *reinterpret_cast<float(*)[32]>(s));
        umma::ld_32x32b_x32(lane_base + kSCol + sb * kSub + 32, s_hi);
        umma::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) s[32 + j] = s_hi[j];
      }
      umma::fence_before_sync();
      arrive_w(kSFree0 + sb);
      const int n_valid = min(kSub, x.t_end - (x.t_begin + i * kSub));
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kSub; ++j) {
        s[j] = (j < n_valid) ? s[j] * row_scale : -INFINITY;
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
        if constexpr (KT == 1) {  // f16 operands
          const __half2 h = __floats2half2_rn(p0, p1);
          pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
          const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      l = (i == 0) ? sum : fmaf(l, alpha, sum);
      // O is rescaled only when some head's max moved; the PV of the previous
      // tile must have landed first (PV(g) waits for this warp's P(g))
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!wait_w(kODone0 + ((g - 1) & 1), ((g - 1) >> 1) & 1)) return;
        umma::fence_after_sync();
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
      m_used = m_new;
      // P row (64 bf16 = 128 bytes) into the 128-byte-swizzled K-major tile
      // inside this tile's stage (S(g), the last reader of those K dims, is done)
      uint8_t* prow = c.smem + kStageOffset + (g % kStages) * kStageBytes +
                      p_offset_in_stage(x.half) + row * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(prow + ((cc ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async();
      umma::fence_before_sync();
      arrive_w(kPFull0 + sb);
      if (i == n_sub - 1) {
        // All S MMAs of this unit are done (S of the last tile was read), so
        // TMEM columns [0, 128) are free: load the next unit's Q now and let
        // the MMA thread start on it while this unit's epilogue runs.
        for (int u2 = next_unit(u); u2 < n_units; u2 = next_unit(u2)) {
          const MlaUnit x2 = mla_unit(p, u2);
          if (x2.empty) continue;
          if (!wait_w(kQFree, n_ne & 1)) return;
          umma::fence_after_sync();
          if (!load_q(x2.b, (n_ne + 1) & 1, e_next)) return;
          q_ready = true;
          break;
        }
      }
    }
    // epilogue: O / l for this half of the value dims
    if (!wait_w(kODone0 + ((g - 1) & 1), ((g - 1) >> 1) & 1)) return;
    umma::fence_after_sync();
    // (an E4M3 cache's value scale multiplies the output once, here)
    const float inv = ((l > 0.f) ? 1.f / l : 0.f) * (KT ? p.v_scale : 1.f);
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
          // partials in the head-interleaved layout (4-dim groups, heads
          // innermost): a warp's store covers 32 consecutive heads, 512 bytes
          const int c0 = (x.half * kDvHalf + ch * 32) / 4;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(p.o_part)[((size_t)x.slot * 128 + c0 + v) * p.H_q + row] =
                make_float4(o[4 * v] * inv, o[4 * v + 1] * inv, o[4 * v + 2] * inv,
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

// ---------------------------------------------------------------- converter
// E4M3 cache only: warps 10-13.  Per tile, once its raw bytes have landed,
// thread t widens the bytes 96 (t % 2) .. + 95 of row t / 2's three pieces
// (six 16-byte runs of 16 dims each) into the row's 16-byte f16 chunks,
// 128-byte-swizzled: piece 0 first (f16 regions 0..2, below the raw bytes),
// then it reads pieces 1 and 2, meets the other three warps at a named
// barrier and writes regions 3..8 (see the E4M3 note at the top).  The four
// warps decide together whether to go on (a bounded wait that ran out in one
// of them ends all four), so none is ever left at the barrier.
__device__ void converter(const Launch& p, const Ctx& c, int n_units) {
  const int ct = threadIdx.x - 320;  // 0..127
  const int lane = ct & 31;
  const int row = ct >> 1, hh = ct & 1;
  uint32_t g = 0;
  for (int u = blockIdx.x; u < n_units; u = next_unit(u)) {
    const MlaUnit x = mla_unit(p, u);
    if (x.empty) continue;
    const int n_sub = (x.t_end - x.t_begin + kSub - 1) / kSub;
    for (int i = 0; i < n_sub; ++i, ++g) {
      const int stage = g % kStages;
      int ok = 1;
      if (lane == 0) ok = wait_bar(c, kRawFull0 + stage, (g / kStages) & 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (named_bar_or(kConvBar, 128, ok == 0)) return;
      uint8_t* st = c.smem + kStageOffset + stage * kStageBytes;
      const uint8_t* raw = st + kRawInStage + row * kRawPiece + hh * 96;
      uint8_t* dst = st + row * 128;
      // 16 E4M3 bytes of dims d0 .. d0 + 15 (d0 a multiple of 16) -> two f16 chunks
      auto put = [&](int d0, uint4 v) {
        uint8_t* rd = dst + (d0 >> 6) * kStageRegion;
        const int k0 = (d0 & 63) >> 3;
        *reinterpret_cast<uint4*>(rd + ((k0 ^ (row & 7)) << 4)) =
            make_uint4(e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y),
                       e4m3x2_to_f16x2(v.y >> 16));
        *reinterpret_cast<uint4*>(rd + (((k0 + 1) ^ (row & 7)) << 4)) =
            make_uint4(e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w),
                       e4m3x2_to_f16x2(v.w >> 16));
      };
#pragma unroll
      for (int q = 0; q < 6; ++q)
        put(96 * hh + 16 * q, *reinterpret_cast<const uint4*>(raw + 16 * q));
      uint4 rv[2][6];
#pragma unroll
      for (int cc = 1; cc < kRawPieces; ++cc)
#pragma unroll
        for (int q = 0; q < 6; ++q)
          rv[cc - 1][q] = *reinterpret_cast<const uint4*>(raw + cc * kRawPieceBytes + 16 * q);
      named_bar_sync(kConvBar, 128);  // every raw byte of the tile is read
#pragma unroll
      for (int cc = 1; cc < kRawPieces; ++cc)
#pragma unroll
        for (int q = 0; q < 6; ++q) put(kRawPiece * cc + 96 * hh + 16 * q, rv[cc - 1][q]);
      fence_proxy_async();  // the MMAs read the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(c, kFull0 + stage));
    }
  }
}

template <int KT>
__global__ void __launch_bounds__(threads_for<KT>(), 1)
    split_mla_kernel(Launch p,
                     const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
  c.hdr = p.hdr;
  c.tm_q = &tm_q;
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
      if ((i >= kSFree0 && i < kSFree0 + 2) || (i >= kPFull0 && i < kPFull0 + 2) ||
          i == kOFree || i == kQTFull)
        count = 4;                                                   // softmax warps
      if (i == kDrain) count = 2;                                    // the two issuing threads
      // a stage's copies: one cp.async arrival per producer thread (E4M3
      // cache: on the raw barrier; kFull then counts the converter warps)
      if (i >= kFull0 && i < kFull0 + kStages) count = KT ? 4 : 128;
      if (KT == 1 && i >= kRawFull0 && i < kRawFull0 + kStages) count = 128;
      mbar_init(bar_addr(c, i), count);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    umma::tmem_alloc(c.sbase + kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  // the barriers exist before any role copies into or arrives on them
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

  // tiles whose P.V and units whose S MMAs the issuing threads got through
  volatile uint32_t* done = reinterpret_cast<volatile uint32_t*>(smem + kAbortSlot + 4);
  if (warp < 4) {
    softmax_warps<KT>(p, c, tmem, n_units);
  } else if (warp < 8) {
    producer<KT>(p, c, n_units);
  } else if (warp >= 10) {
    if constexpr (KT == 1) converter(p, c, n_units);
  } else if ((threadIdx.x & 31) == 0) {
    uint32_t count = 0;
    if (warp == 8)
      mma_s<KT>(p, c, tmem, n_units, count);
    else
      mma_pv<KT>(p, c, tmem, n_units, count);
    done[warp - 8] = count;
    // drain (one commit per issuing thread): its arrival means every MMA the
    // thread issued has completed, so tensor memory can be freed
    umma::commit(bar_addr(c, kDrain));
  }
  umma::fence_before_sync();
  __syncthreads();
  const uint32_t q_done = done[0], g_done = done[1];
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
    // the last releases of the stages and of Q (commits issued before the
    // drain): wait until they have landed, so no arrive is still in flight
    // when the shared memory is given up
    if ((threadIdx.x & 31) == 0) {
      for (int st = 0; st < kStages; ++st) {
        const int last = (int)g_done - 1 - (((int)g_done - 1 - st) % kStages + kStages) % kStages;
        if (last >= 0 && !mbar_wait(bar_addr(c, kEmpty0 + st), (last / kStages) & 1))
          set_error(p.hdr, DA_DEVERR_TIMEOUT);
      }
      if (q_done > 0 && !mbar_wait(bar_addr(c, kQFree), (q_done - 1) & 1))
        set_error(p.hdr, DA_DEVERR_TIMEOUT);
    }
    __syncwarp();
    umma::tmem_dealloc(tmem, kTmemCols);
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

// `rows` rows of 576 bf16 at `base` (16-byte aligned), box {64, box_rows},
// 128-byte swizzle.
bool encode_rows(CUtensorMap* tm, const void* base, long long rows, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || rows < 1 || rows > (1ll << 32)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDqk * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KT>
cudaError_t set_smem() {
  static const cudaError_t e = cudaFuncSetAttribute(
      split_mla_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

}  // namespace

bool mla_supported(int H_q) { return H_q >= 16 && H_q <= kHeads; }

// Persistent CTAs: as many as can be resident at once (one per SM: both
// instantiations take nearly all of the shared memory), rounded down to an
// even number (units are dealt to pairs of CTAs).
int mla_resident_ctas(int sms) {
  static const int per_sm = [] {
    if (set_smem<0>() != cudaSuccess) return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, split_mla_kernel<0>, threads_for<0>(),
                                                      kSmemBytes) != cudaSuccess || n < 1)
      n = 1;
    return n;
  }();
  const int n = per_sm * sms;
  return n < 2 ? 2 : (n & ~1);
}

cudaError_t launch_split_mla(const Launch& p, int grid, cudaStream_t stream) {
  // bf16 or E4M3 (kv_type 0 or 1; E4M3 with one source)
  const int kt = p.kv_type;
  if (kt < 0 || kt > 1 || (kt == 1 && p.extra_k)) return cudaErrorInvalidValue;
  const cudaError_t attr = kt ? set_smem<1>() : set_smem<0>();
  if (attr != cudaSuccess) return attr;
  // rows addressable in the main cache under its layout (none: the kernel
  // reads a zero row for every masked entry instead)
  Launch lp = p;
  lp.kv_rows = (p.layout == DA_KV_CONTIGUOUS) ? (long long)p.B * p.width
               : (p.layout == DA_KV_PAGED)    ? p.num_blocks * p.page_size
                                              : p.num_blocks;
  alignas(64) CUtensorMap tm_q;
  memset(&tm_q, 0, sizeof tm_q);
  if ((long long)p.B * p.H_q >= kQBoxRows &&
      !encode_rows(&tm_q, p.q, (long long)p.B * p.H_q, kQBoxRows))
    return cudaErrorInvalidValue;
  if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;  // whole pairs only
  if (kt == 1)
    return launch_after(split_mla_kernel<1>, dim3(grid), dim3(threads_for<1>()),
                        (size_t)kSmemBytes, stream, lp, tm_q);
  return launch_after(split_mla_kernel<0>, dim3(grid), dim3(threads_for<0>()), (size_t)kSmemBytes,
                      stream, lp, tm_q);
}

}  // namespace da
