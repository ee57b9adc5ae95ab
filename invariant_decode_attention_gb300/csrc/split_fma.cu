// Split kernel, CUDA-core variant (any number of query heads per KV head;
// head dim 64 or 128).
//
// One unit of work = (row b, split s, KV head h, head chunk c): up to Gc
// query heads of group h (chunk c of the group; Gc = 1, 2, 4 or 8 with
// Gc * D <= 512, fixed by the head config) attend over the split's tiles of
// row b's KV list and produce either the row's final output (single-split
// rows) or an fp32 partial (out, lse) that the combine merges.  A group of
// G heads is cut into ceil(G / Gc) chunks; slots of the last chunk past the
// group's end compute on a zero query and are never written.  The chunks of
// one KV head are consecutive units, so they run at the same time on
// neighbouring CTAs and their second reads of K and V come from L2.  Work
// placement is persistent: which CTA runs a unit never changes what the unit
// computes.
//
// Inside a CTA, four warps share each unit.  Warp w owns entries
// [16w, 16w + 16) of every 64-entry tile and streams exactly those K and V
// rows with 16-byte cp.async into its own three-slot shared-memory ring, so
// a warp never waits for another warp inside the tile loop.  Eight lanes
// share an entry (two 16-byte chunks of a 128-dim row each), so a score is an
// 8-lane butterfly sum, and a lane keeps fp32 accumulators for the G heads
// over its own dims, as packed pairs updated with two-wide FMAs.  Online
// softmax runs in the log2 domain with a warp-uniform running max.  At the end
// of a unit the lane groups and then the warps merge in a fixed order.  Every reduction has a fixed shape and order,
// so a unit's bits depend only on its inputs and its split boundaries.
//
// Softmax attention and its split/merge are the computation the FlashMLA
// issue #212 page ("Sparse MLA decode is not batch-invariant") reports on; the
// kernel design here is this library's own.
#include "common.cuh"

namespace da {
namespace {

// Element types of the K and V caches (template argument KT).
enum KvType {
  kKvBf16 = 0,  // bf16
  kKvE4m3 = 1,  // one E4M3 byte per element (DA_KV_FP8_E4M3)
  kKvFp4 = 2,   // E2M1 codes, two per byte, one E4M3 scale per 16 (DA_KV_NVFP4)
};

template <int G, int D, int KT = kKvBf16>
struct FmaShape {
  static constexpr int kTile = kFmaTile;               // entries per tile
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTokPerWarp = kTile / kWarps;    // 16
  static constexpr int kSteps = kTokPerWarp / 4;        // 4 entries per warp step
  static constexpr int kChunks = D / 64;                // 16-byte chunks per lane per row
  static constexpr int kDpl = kChunks * 8;              // dims per lane
  static constexpr int kStages = 3;                     // ring slots per warp
  // bytes of one head's row of codes (and, for kKvFp4, of its block scales)
  static constexpr int kRowBytes = KT == kKvBf16 ? D * 2 : KT == kKvE4m3 ? D : D / 2;
  static constexpr int kScaleRowBytes = KT == kKvFp4 ? D / 16 : 0;
  // 16-byte copies per lane per row (8 lanes per row; a shorter row is copied
  // by the lanes 0 .. kRowBytes / 16 - 1 of the group)
  static constexpr int kCopies = (kRowBytes + 127) / 128;
  // K (or V) of one warp: 16 rows of codes, then (kKvFp4) 16 rows of scales
  static constexpr int kScalesOffset = kTokPerWarp * kRowBytes;
  static constexpr int kSliceBytes = kScalesOffset + kTokPerWarp * kScaleRowBytes;
  static_assert(kSliceBytes % 16 == 0, "slices stay 16-byte aligned");
  static constexpr int kWarpSlotBytes = 2 * kSliceBytes;
  static constexpr int kRingBytes = kStages * kWarps * kWarpSlotBytes;
  static constexpr int kQBytes = G * D * 2;
  static constexpr int kQPad = (kQBytes + 127) / 128 * 128;
  static constexpr int kQOffset = kRingBytes;
  static constexpr int kScratchOffset = kQOffset + kStages * kQPad;
  // Per (warp, head) merge record: D accumulators, then m and l; rows padded
  // to a multiple of 4 floats so float4 stores stay 16-byte aligned.
  static constexpr int kSRow = D + 4;
  static constexpr int kScratchFloats = kWarps * G * kSRow;
  static constexpr int kSmemBytes = kScratchOffset + kScratchFloats * 4;
  static constexpr int kQChunks = kQBytes / 16;         // 16-byte chunks of a query group
  static_assert(D % 64 == 0, "head dim must be a multiple of 64");
  static_assert(kQChunks <= kThreads, "one q chunk per thread at most");
};

// The reference value the exponentials are taken against moves only when a
// score exceeds it by more than 2^8 (log2 units): a warp then reduces the
// tile maxima and rescales; otherwise p <= 2^8 is formed against the old
// value with no cross-lane reduction.  The decision depends only on the
// unit's own scores, so it is the same in every batch.
constexpr float kRescaleLog2 = 8.f;

// A work unit as the kernel sees it: the plan's item descriptor plus a KV
// head and a chunk of its query heads.
struct Unit {
  int slot, tb, te, L, b, h;
  int hq0;     // first query head of the chunk
  int live;    // query heads of the chunk inside the group (the rest are padding)
  int l_main;  // entries before the second source starts
  bool single;
};

// Units per (row, split) item: one per KV head and head chunk.
__device__ __forceinline__ int units_per_item(const Launch& p) {
  return p.H_kv * p.fma_chunks;
}

__device__ __forceinline__ int4 load_desc(const Launch& p, int u) {
  return __ldg(reinterpret_cast<const int4*>(p.item_desc) + u / units_per_item(p));
}

// X: the call has a second KV source (a separate instantiation, so that the
// single-source loop carries none of its checks).
template <int Gc, bool X>
__device__ __forceinline__ Unit make_unit(const Launch& p, int u, int4 d) {
  Unit x;
  x.single = d.x < 0;
  x.slot = x.single ? ~d.x : d.x;
  x.tb = d.y;
  x.te = d.z;
  x.L = d.w;
  x.b = x.slot / p.max_splits;
  const int r = u % units_per_item(p), c = r % p.fma_chunks;
  x.h = r / p.fma_chunks;
  x.hq0 = x.h * p.fma_group + c * Gc;
  x.live = min(Gc, p.fma_group - c * Gc);
  x.l_main = X ? clamp_len(__ldg(p.lengths + x.b), p.capacity) : 0x7fffffff;
  return x;
}

// Cache row (in units of [H_kv, D] records) holding entry `tok` of row b;
// entries from l_main on come from the second source (*src = 1).
template <bool X>
__device__ __forceinline__ bool entry_row(const Launch& p, int b, int tok, int l_main,
                                          long long* row, int* src) {
  *src = 0;
  if (X && tok >= l_main) {
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

// Work queue.  Units with tiles are taken in work-list order (largest first).
// While every CTA still has a full round, CTA c takes unit k * grid + c in
// round k: the KV heads of one item (consecutive units) then run at the same
// time on neighbouring CTAs and read the same cache records together.  The
// remaining units -- less than one round -- come from an atomic counter in the
// workspace header, so the CTAs that finish first take them.  Thread 0 takes
// ids kAhead units ahead into a ring in shared memory (kRing slots).  While the compute works
// on tile t of unit ordinal o, a warp's prefetch cursor has loaded tile t + 2
// and stands on tile t + 3 -- at most ordinal o + 3 when units have one tile
// -- and reads the id of the ordinal after it, o + 4: ids up to o + 4 must be
// known, so the ring is filled five ahead (and slot o + 5 - kRing = o - 3,
// long finished, is the one reused).  Which CTA runs a unit never changes
// what the unit computes.
constexpr int kRing = 8;
constexpr int kAhead = 5;
static_assert(kAhead < kRing - 2, "the reused slot is behind the compute");

// The unit id of this CTA's ordinal `ord` (ids >= n_units: no more work).
__device__ __forceinline__ int unit_of(const Launch& p, int ord, int n_static) {
  const int s = ord * (int)gridDim.x + (int)blockIdx.x;
  return (s < n_static) ? s : n_static + atomicAdd(p.hdr + kHdrQueue, 1);
}

// Position of the prefetch stream: a (unit, tile) pair; ord is the unit's
// ordinal in this CTA's sequence.  The descriptor of the next unit is loaded
// one unit ahead.  In the PF instantiation (a paged cache whose pages hold 16
// or 32 entries, so that the four warps' slices of a tile lie in different
// pages or page halves) the page of this warp's slice is loaded as soon as
// the cursor stands on the tile, a whole slice before its copies are issued;
// otherwise load_slice looks it up itself.
struct Cursor {
  Unit x;
  int ord, k;
  int4 next;
  int page;  // page-table entry of the warp's slice (when `paged` is set)
  bool valid, paged;
};

template <int Gc, bool X>
__device__ __forceinline__ void cursor_seek(const Launch& p, Cursor& c, int ord, int4 d,
                                            const volatile int* ring, int n_units) {
  const int u = ring[ord % kRing];
  if (u >= n_units) {
    c.valid = false;
    return;
  }
  const int un = ring[(ord + 1) % kRing];
  c.next = (un < n_units) ? load_desc(p, un) : make_int4(0, 0, 0, 0);
  c.ord = ord;
  c.x = make_unit<Gc, X>(p, u, d);
  c.k = c.x.tb;
  c.valid = true;
}

template <int Gc, bool X>
__device__ __forceinline__ void cursor_next(const Launch& p, Cursor& c, const volatile int* ring,
                                            int n_units) {
  if (!c.valid) return;
  if (++c.k < c.x.te) return;
  cursor_seek<Gc, X>(p, c, c.ord + 1, c.next, ring, n_units);
}

// PF: load the page of warp `warp`'s slice of the cursor's tile when every
// live entry of the slice sits in one page of the main source (then the page
// table is the slice's only address lookup).
template <bool X, bool PF>
__device__ __forceinline__ void cursor_page(const Launch& p, Cursor& c, int warp) {
  c.paged = false;
  if (!PF || !c.valid || p.layout != DA_KV_PAGED || (p.page_size & 15) != 0) return;
  const int t0 = c.k * kFmaTile + warp * (kFmaTile / 4);
  if (t0 >= c.x.L || (X && min(t0 + kFmaTile / 4, c.x.L) > c.x.l_main)) return;
  const int pi = (p.page_shift >= 0) ? (t0 >> p.page_shift) : (t0 / p.page_size);
  c.page = __ldg(p.table + (size_t)c.x.b * p.width + pi);
  c.paged = true;
}

// Issue this warp's copies for the cursor's tile into ring slot `slot`, then
// close the cp.async group (always, so group counting stays uniform).
template <int G, int D, bool X, int KT, bool PF>
__device__ __forceinline__ void load_slice(const Launch& p, const Cursor& c, uint8_t* smem,
                                           int slot, int warp, int lane) {
  using S = FmaShape<G, D, KT>;
  if (c.valid) {
    const int grp = lane >> 3, sub = lane & 7;
    uint8_t* ks = smem + (slot * S::kWarps + warp) * S::kWarpSlotBytes;
    uint8_t* vs = ks + S::kSliceBytes;
    const int t0 = c.k * S::kTile + warp * S::kTokPerWarp;  // a multiple of 16
    // Contiguous rows, and pages of a multiple of 16 entries, put the warp's
    // 16 entries in consecutive cache rows: one page lookup per slice.
    bool uniform = false, base_ok = true;
    long long base_row = 0;
    // (only when every live entry of the slice comes from the main source)
    if (t0 < c.x.L && (!X || min(t0 + S::kTokPerWarp, c.x.L) <= c.x.l_main)) {
      if (p.layout == DA_KV_CONTIGUOUS) {
        uniform = true;
        base_row = (long long)c.x.b * p.width + t0;
      } else if (PF && c.paged) {  // the page was loaded when the cursor reached the slice
        uniform = true;
        const int pi = (p.page_shift >= 0) ? (t0 >> p.page_shift) : (t0 / p.page_size);
        base_ok = c.page >= 0 && c.page < p.num_blocks;
        base_row = (long long)c.page * p.page_size + (t0 - pi * p.page_size);
      } else if (!PF && p.layout == DA_KV_PAGED && (p.page_size & 15) == 0) {
        uniform = true;
        const int pi = (p.page_shift >= 0) ? (t0 >> p.page_shift) : (t0 / p.page_size);
        const int page = __ldg(p.table + (size_t)c.x.b * p.width + pi);
        base_ok = page >= 0 && page < p.num_blocks;
        base_row = (long long)page * p.page_size + (t0 - pi * p.page_size);
      }
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < S::kSteps; ++j) {
      const int tl = 4 * j + grp;
      const int tok = t0 + tl;
      if (tok < c.x.L) {
        long long row = base_row + tl;
        int src = 0;
        const bool ok = uniform ? base_ok : entry_row<X>(p, c.x.b, tok, c.x.l_main, &row, &src);
        bad |= !ok;
        if (ok) {
          // byte offset of the row of KV head h
          const size_t off = ((size_t)row * p.H_kv + c.x.h) * S::kRowBytes;
          const char* kb = reinterpret_cast<const char*>((X && src) ? p.extra_k : p.k);
          const char* vb = reinterpret_cast<const char*>((X && src) ? p.extra_v : p.v);
#pragma unroll
          for (int ch = 0; ch < S::kCopies; ++ch) {
            const int e = (sub + 8 * ch) * 16;  // byte offset of this 16-byte copy
            if (S::kRowBytes % 128 != 0 && e >= S::kRowBytes) continue;
            cp_async16(smem_addr(ks + tl * S::kRowBytes + e), kb + off + e);
            cp_async16(smem_addr(vs + tl * S::kRowBytes + e), vb + off + e);
          }
          if constexpr (KT == kKvFp4) {
            // the row's block scales sit in the scale region after all codes
            if (sub == 7) {
              const size_t so = (size_t)p.kv_rows * p.H_kv * S::kRowBytes +
                                ((size_t)row * p.H_kv + c.x.h) * S::kScaleRowBytes;
              const uint32_t kd = smem_addr(ks + S::kScalesOffset + tl * S::kScaleRowBytes);
              const uint32_t vd = smem_addr(vs + S::kScalesOffset + tl * S::kScaleRowBytes);
              if constexpr (S::kScaleRowBytes == 8) {
                cp_async8(kd, kb + so);
                cp_async8(vd, vb + so);
              } else {
                cp_async4(kd, kb + so);
                cp_async4(vd, vb + so);
              }
            }
          }
        }
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(p.hdr, DA_DEVERR_INDEX);
    if (c.k == c.x.tb) {
      // the unit's query heads: one 16-byte piece per thread of the CTA;
      // padding slots past the group's end get zeros
      const int id = warp * 32 + lane;
      if (id < S::kQChunks) {
        uint8_t* dst = smem + S::kQOffset + slot * S::kQPad + id * 16;
        if (id / (D / 8) < c.x.live) {
          const __nv_bfloat16* q = p.q + ((size_t)c.x.b * p.H_q + c.x.hq0) * D;
          cp_async16(smem_addr(dst), q + id * 8);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  cp_async_commit();
}

// A lane's dims of one row as packed fp32 pairs: pair 4c + e holds dims
// 64c + 8*sub + 2e and 64c + 8*sub + 2e + 1.
template <int D>
__device__ __forceinline__ void unpack_row2(const uint8_t* row, int sub, uint64_t* f) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint4 w = reinterpret_cast<const uint4*>(row)[sub + 8 * c];
    f[c * 4 + 0] = bf16x2_to_f2(w.x);
    f[c * 4 + 1] = bf16x2_to_f2(w.y);
    f[c * 4 + 2] = bf16x2_to_f2(w.z);
    f[c * 4 + 3] = bf16x2_to_f2(w.w);
  }
}

// The same for an E4M3 row: 8 bytes per lane per 64 dims, each byte converted
// exactly to fp32 (E4M3 values are all representable in f16, and f16 in fp32).
template <int D>
__device__ __forceinline__ void unpack_row2_f8(const uint8_t* row, int sub, uint64_t* f) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint2 w = reinterpret_cast<const uint2*>(row)[sub + 8 * c];
    const uint32_t words[2] = {w.x, w.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const unsigned short two = (unsigned short)(words[h] >> (16 * e));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
        const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
        f[c * 4 + h * 2 + e] = pack2(__low2float(hv), __high2float(hv));
      }
    }
  }
}

// The same for an NVFP4 row: 4 code bytes per lane per 64 dims (8 E2M1
// values, low nibble first) and the lane's block scale (dims 16k .. 16k + 15
// share byte k of the scale row).  Each code becomes an f16 exactly, the f16
// product with the E4M3 scale is exact too (at most 2 x 4 significant bits,
// magnitudes 2^-10 .. 2688), and f16 widens to fp32 exactly.
template <int D>
__device__ __forceinline__ void unpack_row2_fp4(const uint8_t* row, const uint8_t* scales,
                                                int sub, uint64_t* f) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(row)[sub + 8 * c];
    const uint32_t s2 = e4m3x2_to_f16x2(scales[4 * c + (sub >> 1)]);
    const uint32_t sc = __byte_perm(s2, 0, 0x1010);  // (s, s)
    uint32_t hv[4];
    e2m1x8_to_f16x2(w, hv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t h2 = hmul2(hv[e], sc);
      const __half2 hp = *reinterpret_cast<const __half2*>(&h2);
      f[c * 4 + e] = pack2(__low2float(hp), __high2float(hp));
    }
  }
}

// Row `r` of a slice (K or V part) as the lane's packed fp32 pairs.
template <int G, int D, int KT>
__device__ __forceinline__ void unpack_kv2(const uint8_t* part, int r, int sub, uint64_t* f) {
  using S = FmaShape<G, D, KT>;
  if constexpr (KT == kKvE4m3)
    unpack_row2_f8<D>(part + r * S::kRowBytes, sub, f);
  else if constexpr (KT == kKvFp4)
    unpack_row2_fp4<D>(part + r * S::kRowBytes, part + S::kScalesOffset + r * S::kScaleRowBytes,
                       sub, f);
  else
    unpack_row2<D>(part + r * S::kRowBytes, sub, f);
}

// Lane-dependent orders that let the 8 lanes of an entry group reduce their
// partial dot products by halving (each level: v[i] += shfl_xor(v[i + half]))
// with no data-dependent selects.  For G >= 2 a lane with sub-lane bits
// (b2 b1 b0) keeps, in entry slot js, the entry js ^ tperm and, in head slot
// hs, the head hs ^ hperm:
//     tperm = 2*b2 + b1,  hperm = b0 * G/2.
// The permutation is applied where rows are addressed (K, V, q, outputs);
// values in registers are never shuffled into place.  For G == 1 both are 0
// and an 8-lane butterfly is used instead.
template <int G>
__device__ __forceinline__ int tperm_of(int sub) {
  return G >= 2 ? (((sub >> 2) & 1) << 1 | ((sub >> 1) & 1)) : 0;
}
template <int G>
__device__ __forceinline__ int hperm_of(int sub) {
  return G >= 2 ? (sub & 1) * (G / 2) : 0;
}

// One warp's 16 entries of one tile: scores, online-softmax update, P.V.
// Dot products and the P.V update use packed fp32 pairs (two FMAs per
// instruction); a partial score is the sum of its even-dim and odd-dim halves.
//
// G >= 2: after the halving reduction a lane holds the full scores of its own
// entry (slot 0) for head slots 0 .. G/2-1.  l[i] (i < G/2) sums p over the
// lane's own entries only; lanes are summed at the end of the unit.
// G == 1: every lane of a group ends with the group's scores (butterfly) and
// l[0] counts the group's entries.
template <int G, int D, int KT, bool kPartial>
__device__ __forceinline__ void consume_slice(const uint8_t* ks, int lane, int n_valid,
                                              const uint64_t (&q2)[G][FmaShape<G, D>::kDpl / 2],
                                              float (&m)[G], float (&l)[G],
                                              uint64_t (&acc2)[G][FmaShape<G, D>::kDpl / 2],
                                              float scale_log2) {
  using S = FmaShape<G, D, KT>;
  constexpr int kP = S::kDpl / 2;  // packed pairs per lane
  constexpr int kV = S::kSteps * G;  // partial scores per lane
  const int grp = lane >> 3, sub = lane & 7;
  const int tp = tperm_of<G>(sub);
  const uint8_t* vs = ks + S::kSliceBytes;

  // ---- partial scores v[js * G + hs] over this lane's dims
  float v[kV];
#pragma unroll
  for (int js = 0; js < S::kSteps; ++js) {
    uint64_t k2[kP];
    unpack_kv2<G, D, KT>(ks, 4 * (js ^ tp) + grp, sub, k2);
#pragma unroll
    for (int hs = 0; hs < G; ++hs) {
      uint64_t a = ffma2(q2[hs][0], k2[0], 0ull);
#pragma unroll
      for (int i = 1; i < kP; ++i) a = ffma2(q2[hs][i], k2[i], a);
      float lo, hi;
      unpack2(a, lo, hi);
      v[js * G + hs] = lo + hi;
    }
  }

  float alpha[G];
  bool rescale = false;
  float pfull[S::kSteps][G];  // p of entry slot js, head slot hs
  if constexpr (G >= 2) {
    // ---- halving reduction over the 8 lanes of the group
#pragma unroll
    for (int i = 0; i < kV / 2; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + kV / 2], 4);
#pragma unroll
    for (int i = 0; i < kV / 4; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + kV / 4], 2);
#pragma unroll
    for (int i = 0; i < kV / 8; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + kV / 8], 1);
    // v[0 .. G/2-1]: own entry (4 * tp + grp), head slots 0 .. G/2-1
    const bool own_valid = !kPartial || (4 * tp + grp) < n_valid;
    float sc[G / 2];
    bool jump = false;  // some score exceeds its running max by more than 2^8
#pragma unroll
    for (int i = 0; i < G / 2; ++i) {
      sc[i] = own_valid ? v[i] * scale_log2 : -INFINITY;
      jump |= sc[i] > m[i] + kRescaleLog2;
    }
    float mnew[G];
    if (__any_sync(0xffffffffu, jump)) {
      // the slow path: the tile maxima of every head, then the standard
      // online-softmax update (the reference value becomes the running max)
      float tmax[G];
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        float mx = sc[i];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        tmax[i] = mx;
      }
#pragma unroll
      for (int i = 0; i < G / 2; ++i) tmax[i + G / 2] = __shfl_xor_sync(0xffffffffu, tmax[i], 1);
#pragma unroll
      for (int hs = 0; hs < G; ++hs) {
        mnew[hs] = fmaxf(m[hs], tmax[hs]);
        alpha[hs] = (mnew[hs] == -INFINITY) ? 1.f : ex2(m[hs] - mnew[hs]);
        rescale |= (alpha[hs] != 1.f);
        m[hs] = mnew[hs];
      }
    } else {
      // every score is at most 2^8 above its head's reference value: keep it
#pragma unroll
      for (int hs = 0; hs < G; ++hs) {
        mnew[hs] = m[hs];
        alpha[hs] = 1.f;
      }
    }
    // ---- own probabilities, own share of l
    float pown[G / 2];
#pragma unroll
    for (int i = 0; i < G / 2; ++i) {
      pown[i] = (mnew[i] == -INFINITY) ? 0.f : ex2(sc[i] - mnew[i]);
      l[i] = fmaf(l[i], alpha[i], pown[i]);
    }
    // ---- all-gather p to the 8 lanes of the group (reverse of the halving)
#pragma unroll
    for (int i = 0; i < G / 2; ++i) {
      pfull[0][i] = pown[i];
      pfull[0][i + G / 2] = __shfl_xor_sync(0xffffffffu, pown[i], 1);
    }
#pragma unroll
    for (int hs = 0; hs < G; ++hs) pfull[1][hs] = __shfl_xor_sync(0xffffffffu, pfull[0][hs], 2);
#pragma unroll
    for (int js = 0; js < 2; ++js)
#pragma unroll
      for (int hs = 0; hs < G; ++hs)
        pfull[js + 2][hs] = __shfl_xor_sync(0xffffffffu, pfull[js][hs], 4);
  } else {
    // ---- G == 1: 8-lane butterfly, every lane of the group gets the sums
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
      for (int i = 0; i < kV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
    bool jump = false;  // some score exceeds the running max by more than 2^8
#pragma unroll
    for (int js = 0; js < S::kSteps; ++js) {
      const bool valid = !kPartial || (4 * js + grp) < n_valid;
      v[js] = valid ? v[js] * scale_log2 : -INFINITY;
      jump |= v[js] > m[0] + kRescaleLog2;
    }
    float mn = m[0];
    alpha[0] = 1.f;
    if (__any_sync(0xffffffffu, jump)) {
      float mx = -INFINITY;
#pragma unroll
      for (int js = 0; js < S::kSteps; ++js) mx = fmaxf(mx, v[js]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      mn = fmaxf(m[0], mx);
      alpha[0] = (mn == -INFINITY) ? 1.f : ex2(m[0] - mn);
      rescale = alpha[0] != 1.f;
      m[0] = mn;
    }
    float sum = 0.f;
#pragma unroll
    for (int js = 0; js < S::kSteps; ++js) {
      pfull[js][0] = (mn == -INFINITY) ? 0.f : ex2(v[js] - mn);
      sum += pfull[js][0];
    }
    l[0] = fmaf(l[0], alpha[0], sum);
  }
  if (rescale) {
#pragma unroll
    for (int hs = 0; hs < G; ++hs) {
      const uint64_t a2 = pack2(alpha[hs], alpha[hs]);
#pragma unroll
      for (int i = 0; i < kP; ++i) acc2[hs][i] = fmul2(acc2[hs][i], a2);
    }
  }
  // ---- P.V over the group's 4 entries
#pragma unroll
  for (int js = 0; js < S::kSteps; ++js) {
    const int row = 4 * (js ^ tp) + grp;
    if (kPartial && row >= n_valid) continue;  // never read unfilled rows
    uint64_t v2[kP];
    unpack_kv2<G, D, KT>(vs, row, sub, v2);
#pragma unroll
    for (int hs = 0; hs < G; ++hs) {
      const uint64_t p2 = pack2(pfull[js][hs], pfull[js][hs]);
#pragma unroll
      for (int i = 0; i < kP; ++i) acc2[hs][i] = ffma2(p2, v2[i], acc2[hs][i]);
    }
  }
}

template <int G, int D, bool X, int KT, bool PF>
__global__ void __launch_bounds__(FmaShape<G, D>::kThreads) split_fma_kernel(Launch p) {
  using S = FmaShape<G, D, KT>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* scratch = reinterpret_cast<float*>(smem + S::kScratchOffset);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, sub = lane & 7;
  wait_prior_grid();  // the plan kernel's outputs
  allow_next_grid();
  __shared__ int ring[kRing];  // unit ids of this CTA's ordinals, kAhead ahead
  const int n_items = p.hdr[kHdrNWork], n_empty = p.hdr[kHdrNEmpty];
  const int upi = units_per_item(p);
  const int n_units = (n_items - n_empty) * upi;  // units with tiles, listed first
  // units of empty rows (listed last): out = 0, lse = -inf, dealt round-robin
  for (int e = n_units + blockIdx.x; e < n_items * upi; e += gridDim.x) {
    const Unit x = make_unit<G, false>(p, e, load_desc(p, e));  // an empty row has one split
    for (int i = threadIdx.x; i < x.live * D; i += S::kThreads)
      p.out[((size_t)x.b * p.H_q + x.hq0) * D + i] = __float2bfloat16_rn(0.f);
    if (threadIdx.x < x.live) p.lse[(size_t)x.b * p.H_q + x.hq0 + threadIdx.x] = -INFINITY;
  }
  const int n_static = n_units / (int)gridDim.x * (int)gridDim.x;  // whole rounds
  if (threadIdx.x == 0)
    for (int i = 0; i < kAhead; ++i) ring[i] = unit_of(p, i, n_static);
  __syncthreads();

  // prologue: fill kStages - 1 slots
  Cursor pf;
  if (ring[0] < n_units)
    cursor_seek<G, X>(p, pf, 0, load_desc(p, ring[0]), ring, n_units);
  else
    pf.valid = false;
  cursor_page<X, PF>(p, pf, warp);
#pragma unroll
  for (int s = 0; s < S::kStages - 1; ++s) {
    load_slice<G, D, X, KT, PF>(p, pf, smem, s, warp, lane);
    cursor_next<G, X>(p, pf, ring, n_units);
    cursor_page<X, PF>(p, pf, warp);
  }

  int slot = 0;
  uint64_t q2[G][S::kDpl / 2];
  int4 d_next = (ring[0] < n_units) ? load_desc(p, ring[0]) : make_int4(0, 0, 0, 0);
  for (int ord = 0;; ++ord) {
    const int u = ring[ord % kRing];
    if (u >= n_units) break;
    const Unit x = make_unit<G, X>(p, u, d_next);
    const int un = ring[(ord + 1) % kRing];
    if (un < n_units) d_next = load_desc(p, un);
    float m[G], l[G];
    uint64_t acc2[G][S::kDpl / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < S::kDpl / 2; ++i) acc2[h][i] = 0ull;
    }
    for (int k = x.tb; k < x.te; ++k) {
      cp_async_wait<S::kStages - 2>();
      if (k == x.tb) {
        // the query group was copied by threads of every warp: all four must
        // have waited on their copies before anyone reads it, and all must
        // have read it before any slot holding it can be refilled
        named_bar_sync(1, S::kThreads);
        const uint8_t* sq = smem + S::kQOffset + slot * S::kQPad;
#pragma unroll
        for (int hs = 0; hs < G; ++hs)
          unpack_row2<D>(sq + (hs ^ hperm_of<G>(sub)) * (D * 2), sub, q2[hs]);  // bf16 q
        named_bar_sync(1, S::kThreads);
      }
      // refill the slot consumed in the previous iteration
      load_slice<G, D, X, KT, PF>(p, pf, smem, (slot + S::kStages - 1) % S::kStages, warp,
                                  lane);
      cursor_next<G, X>(p, pf, ring, n_units);
      cursor_page<X, PF>(p, pf, warp);
      const uint8_t* ks = smem + (slot * S::kWarps + warp) * S::kWarpSlotBytes;
      const int n_valid = min(S::kTokPerWarp, x.L - k * S::kTile - warp * S::kTokPerWarp);
      if (n_valid >= S::kTokPerWarp)
        consume_slice<G, D, KT, false>(ks, lane, n_valid, q2, m, l, acc2, p.scale_log2);
      else
        consume_slice<G, D, KT, true>(ks, lane, n_valid, q2, m, l, acc2, p.scale_log2);
      slot = (slot + 1 == S::kStages) ? 0 : slot + 1;
    }

    // ---- merge: lanes within the warp, then warps --------------------------
    // l: G >= 2 sums each lane's own entries (slots 0 .. G/2-1) over the 32
    // lanes that share a head, then hands the other half of the heads over
    // from the neighbouring lane; G == 1 sums the four entry groups.
    if constexpr (G >= 2) {
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 4);
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 8);
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 16);
      }
#pragma unroll
      for (int i = 0; i < G / 2; ++i) l[i + G / 2] = __shfl_xor_sync(0xffffffffu, l[i], 1);
    } else {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 8);
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 16);
    }
    float acc[G][S::kDpl];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < S::kDpl / 2; ++i) unpack2(acc2[h][i], acc[h][2 * i], acc[h][2 * i + 1]);
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) {
        acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], 8);
        acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], 16);
      }
    }
    if (grp == 0) {
      const int hp = hperm_of<G>(sub);
#pragma unroll
      for (int hs = 0; hs < G; ++hs) {
        float* dst = scratch + (warp * G + (hs ^ hp)) * S::kSRow;
#pragma unroll
        for (int c = 0; c < S::kChunks; ++c) {
          float4* d4 = reinterpret_cast<float4*>(dst + sub * 8 + c * 64);
          d4[0] = make_float4(acc[hs][c * 8 + 0], acc[hs][c * 8 + 1], acc[hs][c * 8 + 2], acc[hs][c * 8 + 3]);
          d4[1] = make_float4(acc[hs][c * 8 + 4], acc[hs][c * 8 + 5], acc[hs][c * 8 + 6], acc[hs][c * 8 + 7]);
        }
        if (sub == 0) {  // lane 0: hperm = 0, slot = head
          dst[D] = m[hs];
          dst[D + 1] = l[hs];
        }
      }
    }
    named_bar_sync(1, S::kThreads);
    for (int h = warp; h < x.live; h += S::kWarps) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < S::kWarps; ++w) M = fmaxf(M, scratch[(w * G + h) * S::kSRow + D]);
      float wgt[S::kWarps];
      float lt = 0.f;
#pragma unroll
      for (int w = 0; w < S::kWarps; ++w) {
        const float* src = scratch + (w * G + h) * S::kSRow;
        wgt[w] = (M == -INFINITY) ? 0.f : ex2(src[D] - M);
        lt = fmaf(src[D + 1], wgt[w], lt);
      }
      const int hq = x.hq0 + h;
      const float lse2 = (lt > 0.f) ? M + lg2(lt) : -INFINITY;
#pragma unroll
      for (int r = 0; r < D / 32; ++r) {
        const int d = lane + 32 * r;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < S::kWarps; ++w) o = fmaf(scratch[(w * G + h) * S::kSRow + d], wgt[w], o);
        o = (lt > 0.f) ? o / lt : 0.f;
        if constexpr (KT != kKvBf16) o *= p.v_scale;  // cache scale: once, at the output
        if (x.single)
          p.out[((size_t)x.b * p.H_q + hq) * D + d] = __float2bfloat16_rn(o);
        else
          p.o_part[((size_t)x.slot * p.H_q + hq) * D + d] = o;
      }
      if (lane == 0) {
        if (x.single)
          p.lse[(size_t)x.b * p.H_q + hq] = (lt > 0.f) ? lse2 * kLn2 : -INFINITY;
        else
          p.lse_part[(size_t)x.slot * p.H_q + hq] = lse2;
      }
    }
    // the id of ordinal ord + kAhead; the barrier publishes it
    if (threadIdx.x == 0) ring[(ord + kAhead) % kRing] = unit_of(p, ord + kAhead, n_static);
    named_bar_sync(1, S::kThreads);
  }
  cp_async_wait<0>();  // leave no copy in flight
  // the last CTA to finish resets the queue for the next call on this plan
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.hdr + kHdrExits, 1) == (int)gridDim.x - 1) {
      p.hdr[kHdrQueue] = 0;
      p.hdr[kHdrExits] = 0;
    }
  }
}

template <int G, int D, bool X, int KT, bool PF = false>
cudaError_t launch_x(const Launch& p, int grid, cudaStream_t stream) {
  using S = FmaShape<G, D, KT>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(split_fma_kernel<G, D, X, KT, PF>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (attr != cudaSuccess) return attr;
  return launch_after(split_fma_kernel<G, D, X, KT, PF>, dim3(grid), dim3(S::kThreads),
                      S::kSmemBytes, stream, p);
}

// Instantiations: bf16 with one or two KV sources (one source: also the PF
// form for small pages); E4M3 and NVFP4 caches with one source.
template <int G, int D>
cudaError_t launch_one(const Launch& p, int grid, cudaStream_t stream) {
  if (p.kv_type != kKvBf16) {
    if (p.extra_k) return cudaErrorInvalidValue;
    if (p.kv_type == kKvE4m3) return launch_x<G, D, false, kKvE4m3>(p, grid, stream);
    if (p.kv_type == kKvFp4) return launch_x<G, D, false, kKvFp4>(p, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (p.extra_k) return launch_x<G, D, true, kKvBf16>(p, grid, stream);
  // pages of 16 or 32 entries: the page lookups go one slice ahead
  if (p.layout == DA_KV_PAGED && (p.page_size == 16 || p.page_size == 32))
    return launch_x<G, D, false, kKvBf16, true>(p, grid, stream);
  return launch_x<G, D, false, kKvBf16>(p, grid, stream);
}

template <int G, int D>
int ctas_one() {
  using S = FmaShape<G, D>;
  static int n = [] {
    cudaFuncSetAttribute(split_fma_kernel<G, D, false, kKvBf16, false>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    int c = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, split_fma_kernel<G, D, false, kKvBf16, false>,
                                                      S::kThreads,
                                                      S::kSmemBytes) != cudaSuccess)
      c = 1;
    return c < 1 ? 1 : c;
  }();
  return n;
}

}  // namespace

// Query heads per unit (Gc) and units per KV head for a group of G heads:
// Gc = the power of two >= G, at most 8 for D = 64 and 4 for D = 128 (so that
// a lane's query and accumulator registers stay at <= 64 each).
void fma_chunk_shape(int G, int D, int* gc, int* chunks) {
  const int gmax = (D == 64) ? 8 : 4;
  int g = 1;
  while (g < G && g < gmax) g <<= 1;
  *gc = g;
  *chunks = (G + g - 1) / g;
}

bool fma_supported(int G, int D) {
  return G >= 1 && G <= kFmaMaxGroup && (D == 64 || D == 128);
}

cudaError_t launch_split_fma(const Launch& p0, int grid, cudaStream_t stream) {
  const int G = p0.H_q / p0.H_kv, D = p0.D_qk;
  if (!fma_supported(G, D)) return cudaErrorInvalidValue;
  Launch p = p0;
  int gc = 1;
  fma_chunk_shape(G, D, &gc, &p.fma_chunks);
  p.fma_group = G;
  if (gc == 1 && D == 64) return launch_one<1, 64>(p, grid, stream);
  if (gc == 2 && D == 64) return launch_one<2, 64>(p, grid, stream);
  if (gc == 4 && D == 64) return launch_one<4, 64>(p, grid, stream);
  if (gc == 8 && D == 64) return launch_one<8, 64>(p, grid, stream);
  if (gc == 1 && D == 128) return launch_one<1, 128>(p, grid, stream);
  if (gc == 2 && D == 128) return launch_one<2, 128>(p, grid, stream);
  if (gc == 4 && D == 128) return launch_one<4, 128>(p, grid, stream);
  return cudaErrorInvalidValue;
}

int fma_ctas_per_sm(int G, int D) {
  int gc = 1, chunks = 1;
  fma_chunk_shape(G, D, &gc, &chunks);
  if (gc == 1 && D == 64) return ctas_one<1, 64>();
  if (gc == 2 && D == 64) return ctas_one<2, 64>();
  if (gc == 4 && D == 64) return ctas_one<4, 64>();
  if (gc == 8 && D == 64) return ctas_one<8, 64>();
  if (gc == 1 && D == 128) return ctas_one<1, 128>();
  if (gc == 2 && D == 128) return ctas_one<2, 128>();
  if (gc == 4 && D == 128) return ctas_one<4, 128>();
  return 1;
}

}  // namespace da
