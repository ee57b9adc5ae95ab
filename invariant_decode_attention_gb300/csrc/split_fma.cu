// Split kernel, CUDA-core variant (query groups of 1, 2, 4 or 8 heads per KV
// head; head dim 64 or 128; G * D <= 512).
//
// One unit of work = (row b, split s, KV head h): the G query heads of group
// h attend over the split's tiles of row b's KV list and produce either the
// row's final output (single-split rows) or an fp32 partial (out, lse) that
// the combine merges.  Work placement is persistent: CTA c takes units c,
// c + grid, ...; which CTA runs a unit never changes what the unit computes.
//
// Inside a CTA (warp-specialised):
//   * one producer warp streams each tile's K and V rows (and the query group
//     at a unit's first tile) into a ring of shared-memory stages with bulk
//     asynchronous copies (TMA engine), completing on an mbarrier per stage.
//     Per-row copies serve all three cache layouts: a row of one KV head is
//     D_qk*2 contiguous bytes in each of them.
//   * four consumer warps each own 16 of a tile's 64 entries.  Eight lanes
//     share an entry (16-byte chunks of the row each), so a score is an
//     8-lane butterfly reduction, and a lane keeps fp32 accumulators for the
//     G heads over its own dims.  Online softmax runs in the log2 domain with
//     a warp-uniform running max.
//   * at the end of a unit the lane groups and warps merge in a fixed order.
// Every reduction has a fixed shape and order, so a unit's bits depend only
// on its inputs and its split boundaries.
//
// Softmax attention and the split/merge are the computation the FlashMLA
// issue #212 page ("Sparse MLA decode is not batch-invariant") reports on; the
// kernel design here is this library's own.
#include "common.cuh"

namespace da {
namespace {

// Register cap: two 160-thread CTAs per SM.
constexpr int kFmaMaxRegs = 200;

template <int G, int D>
struct FmaShape {
  static constexpr int kTile = kFmaTile;               // entries per tile
  static constexpr int kWarps = 4;                      // consumer warps
  static constexpr int kThreads = (kWarps + 1) * 32;    // + one producer warp
  static constexpr int kTokPerWarp = kTile / kWarps;    // 16
  static constexpr int kSteps = kTokPerWarp / 4;        // 4 entries per warp step
  static constexpr int kChunks = D / 64;                // 16-byte chunks per lane per row
  static constexpr int kDpl = kChunks * 8;              // dims per lane
  static constexpr int kStages = 3;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kKVBytes = kTile * kRowBytes;    // K (or V) bytes per stage
  static constexpr int kQBytes = G * D * 2;
  static constexpr int kQPad = (kQBytes + 127) / 128 * 128;
  static constexpr int kStageBytes = 2 * kKVBytes + kQPad;
  // Per (warp, head) merge record: D accumulators, then m and l; the row is
  // padded to a multiple of 4 floats so float4 stores stay 16-byte aligned.
  static constexpr int kSRow = D + 4;
  static constexpr int kScratchFloats = kWarps * G * kSRow;
  static constexpr int kBarOffset = kStages * kStageBytes + kScratchFloats * 4;
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + 16;
  // Two CTAs per SM when the q + accumulator registers leave room for it.
  static_assert(kFmaMaxRegs * kThreads * 2 <= 65536, "two CTAs per SM");
  static_assert(D % 64 == 0, "head dim must be a multiple of 64");
  static_assert(kTile == 64, "two entries per producer lane");
};

struct Unit {
  int b, h, slot, L, tb, te;
};

__device__ __forceinline__ Unit decode_unit(const Launch& p, int u) {
  Unit x;
  const int item = u / p.H_kv;
  x.h = u - item * p.H_kv;
  x.slot = p.work[item];
  x.b = x.slot / p.max_splits;
  const int s = x.slot - x.b * p.max_splits;
  x.L = clamp_len(p.lengths[x.b], p.capacity);
  const int32_t* sb = p.split_begin + (size_t)x.b * (p.max_splits + 1);
  x.tb = sb[s];
  x.te = sb[s + 1];
  return x;
}

// Cache row (in units of [H_kv, D] records) holding entry `tok` of row b.
__device__ __forceinline__ bool entry_row(const Launch& p, int b, int tok, long long* row) {
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

// Wait that also gives up when another warp has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

template <int G, int D>
__device__ void producer(const Launch& p, uint8_t* stages, uint64_t* full, uint64_t* empty,
                         volatile int* abort_flag, int n_units) {
  using S = FmaShape<G, D>;
  const int lane = threadIdx.x & 31;
  const uint64_t pol_kv = policy_evict_first();
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
    const Unit x = decode_unit(p, u);
    for (int k = x.tb; k < x.te; ++k) {
      if (!wait_or_abort(smem_addr(&empty[stage]), phase ^ 1, abort_flag)) {
        if (lane == 0) {
          set_error(p.hdr, DA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        ok = false;
        break;
      }
      const int t0 = k * S::kTile;
      const int n_valid = min(S::kTile, x.L - t0);
      long long off[2];
      bool go[2], bad = false;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = lane + 32 * i;
        go[i] = false;
        off[i] = 0;
        if (t < n_valid) {
          long long row;
          go[i] = entry_row(p, x.b, t0 + t, &row);
          bad |= !go[i];
          off[i] = (row * p.H_kv + x.h) * D;
        }
      }
      const unsigned m0 = __ballot_sync(0xffffffffu, go[0]);
      const unsigned m1 = __ballot_sync(0xffffffffu, go[1]);
      if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(p.hdr, DA_DEVERR_INDEX);
      const bool first = (k == x.tb);
      const uint32_t bytes =
          (uint32_t)(__popc(m0) + __popc(m1)) * 2u * S::kRowBytes + (first ? S::kQBytes : 0u);
      const uint32_t bar = smem_addr(&full[stage]);
      if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
      __syncwarp();
      uint8_t* st = stages + (size_t)stage * S::kStageBytes;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (go[i]) {
          const int t = lane + 32 * i;
          bulk_g2s(smem_addr(st + t * S::kRowBytes), p.k + off[i], S::kRowBytes, bar, pol_kv);
          bulk_g2s(smem_addr(st + S::kKVBytes + t * S::kRowBytes), p.v + off[i], S::kRowBytes,
                   bar, pol_kv);
        }
      }
      if (first && lane == 0) {
        const __nv_bfloat16* qsrc = p.q + ((size_t)x.b * p.H_q + (size_t)x.h * G) * D;
        bulk_g2s(smem_addr(st + 2 * S::kKVBytes), qsrc, S::kQBytes, bar, pol_kv);
      }
      ++issued;
      if (++stage == S::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  // Do not leave while copies this warp issued may still be landing: wait
  // (bounded) for the fills of the last stages it used.
  const int pending = min(issued, S::kStages);
  for (int i = 0; i < pending; ++i) {
    if (--stage < 0) {
      stage = S::kStages - 1;
      phase ^= 1;
    }
    mbar_wait(smem_addr(&full[stage]), phase);
  }
}

template <int G, int D, bool kPartial>
__device__ __forceinline__ void consume_tile(const uint8_t* st, int warp, int lane, int n_valid,
                                             const float (&qf)[G][FmaShape<G, D>::kDpl],
                                             float (&m)[G], float (&l)[G],
                                             float (&acc)[G][FmaShape<G, D>::kDpl],
                                             float scale_log2) {
  using S = FmaShape<G, D>;
  const int grp = lane >> 3, sub = lane & 7;
  const uint8_t* sK = st;
  const uint8_t* sV = st + S::kKVBytes;

  float s[S::kSteps][G];
#pragma unroll
  for (int j = 0; j < S::kSteps; ++j) {
    const int t = warp * S::kTokPerWarp + j * 4 + grp;
    const uint4* kr = reinterpret_cast<const uint4*>(sK + t * S::kRowBytes);
    float kf[S::kDpl];
#pragma unroll
    for (int c = 0; c < S::kChunks; ++c) {
      const uint4 w = kr[sub + 8 * c];
      kf[c * 8 + 0] = bf16_lo(w.x); kf[c * 8 + 1] = bf16_hi(w.x);
      kf[c * 8 + 2] = bf16_lo(w.y); kf[c * 8 + 3] = bf16_hi(w.y);
      kf[c * 8 + 4] = bf16_lo(w.z); kf[c * 8 + 5] = bf16_hi(w.z);
      kf[c * 8 + 6] = bf16_lo(w.w); kf[c * 8 + 7] = bf16_hi(w.w);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) a = fmaf(qf[h][i], kf[i], a);
      s[j][h] = a;
    }
  }
  // Sum the 8 lanes of each entry (butterfly: every lane ends with the same bits).
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
    for (int j = 0; j < S::kSteps; ++j)
#pragma unroll
      for (int h = 0; h < G; ++h) s[j][h] += __shfl_xor_sync(0xffffffffu, s[j][h], o);
  }
#pragma unroll
  for (int j = 0; j < S::kSteps; ++j) {
    const bool valid = !kPartial || (warp * S::kTokPerWarp + j * 4 + grp) < n_valid;
#pragma unroll
    for (int h = 0; h < G; ++h) s[j][h] = valid ? s[j][h] * scale_log2 : -INFINITY;
  }
  // Warp-wide running max per head.
  bool rescale = false;
  float alpha[G], mnew[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = s[0][h];
#pragma unroll
    for (int j = 1; j < S::kSteps; ++j) mx = fmaxf(mx, s[j][h]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mnew[h] = fmaxf(m[h], mx);
    alpha[h] = (mnew[h] == -INFINITY) ? 1.f : ex2(m[h] - mnew[h]);
    rescale |= (alpha[h] != 1.f);
    m[h] = mnew[h];
  }
  float pr[S::kSteps][G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < S::kSteps; ++j) {
      pr[j][h] = (mnew[h] == -INFINITY) ? 0.f : ex2(s[j][h] - mnew[h]);
      sum += pr[j][h];
    }
    l[h] = fmaf(l[h], alpha[h], sum);
  }
  if (rescale) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) acc[h][i] *= alpha[h];
  }
#pragma unroll
  for (int j = 0; j < S::kSteps; ++j) {
    const int t = warp * S::kTokPerWarp + j * 4 + grp;
    if (kPartial && t >= n_valid) continue;  // stale shared memory: never touch it
    const uint4* vr = reinterpret_cast<const uint4*>(sV + t * S::kRowBytes);
    float vf[S::kDpl];
#pragma unroll
    for (int c = 0; c < S::kChunks; ++c) {
      const uint4 w = vr[sub + 8 * c];
      vf[c * 8 + 0] = bf16_lo(w.x); vf[c * 8 + 1] = bf16_hi(w.x);
      vf[c * 8 + 2] = bf16_lo(w.y); vf[c * 8 + 3] = bf16_hi(w.y);
      vf[c * 8 + 4] = bf16_lo(w.z); vf[c * 8 + 5] = bf16_hi(w.z);
      vf[c * 8 + 6] = bf16_lo(w.w); vf[c * 8 + 7] = bf16_hi(w.w);
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) acc[h][i] = fmaf(pr[j][h], vf[i], acc[h][i]);
  }
}

template <int G, int D>
__device__ void consumer(const Launch& p, uint8_t* stages, float* scratch, uint64_t* full,
                         uint64_t* empty, volatile int* abort_flag, int n_units) {
  using S = FmaShape<G, D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, sub = lane & 7;
  int stage = 0;
  uint32_t phase = 0;
  float qf[G][S::kDpl];
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit x = decode_unit(p, u);
    float m[G], l[G], acc[G][S::kDpl];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) acc[h][i] = 0.f;
    }
    bool alive = !*abort_flag;
    for (int k = x.tb; k < x.te && alive; ++k) {
      if (!wait_or_abort(smem_addr(&full[stage]), phase, abort_flag)) {
        if (lane == 0) {
          set_error(p.hdr, DA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        alive = false;
        break;
      }
      const uint8_t* st = stages + (size_t)stage * S::kStageBytes;
      if (k == x.tb) {
        const uint8_t* sq = st + 2 * S::kKVBytes;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int c = 0; c < S::kChunks; ++c) {
            const uint4 w = reinterpret_cast<const uint4*>(sq + h * S::kRowBytes)[sub + 8 * c];
            qf[h][c * 8 + 0] = bf16_lo(w.x); qf[h][c * 8 + 1] = bf16_hi(w.x);
            qf[h][c * 8 + 2] = bf16_lo(w.y); qf[h][c * 8 + 3] = bf16_hi(w.y);
            qf[h][c * 8 + 4] = bf16_lo(w.z); qf[h][c * 8 + 5] = bf16_hi(w.z);
            qf[h][c * 8 + 6] = bf16_lo(w.w); qf[h][c * 8 + 7] = bf16_hi(w.w);
          }
      }
      const int n_valid = min(S::kTile, x.L - k * S::kTile);
      if (n_valid == S::kTile)
        consume_tile<G, D, false>(st, warp, lane, n_valid, qf, m, l, acc, p.scale_log2);
      else
        consume_tile<G, D, true>(st, warp, lane, n_valid, qf, m, l, acc, p.scale_log2);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[stage]));
      if (++stage == S::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }

    // ---- merge: lane groups (entries) within the warp, then warps ------------
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
#pragma unroll
      for (int i = 0; i < S::kDpl; ++i) {
        acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], 8);
        acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], 16);
      }
    }
    if (grp == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* dst = scratch + (warp * G + h) * S::kSRow;
#pragma unroll
        for (int c = 0; c < S::kChunks; ++c) {
          float4* d4 = reinterpret_cast<float4*>(dst + sub * 8 + c * 64);
          d4[0] = make_float4(acc[h][c * 8 + 0], acc[h][c * 8 + 1], acc[h][c * 8 + 2], acc[h][c * 8 + 3]);
          d4[1] = make_float4(acc[h][c * 8 + 4], acc[h][c * 8 + 5], acc[h][c * 8 + 6], acc[h][c * 8 + 7]);
        }
        if (sub == 0) {
          dst[D] = m[h];
          dst[D + 1] = l[h];
        }
      }
    }
    named_bar_sync(1, S::kWarps * 32);
    const bool single = p.n_splits[x.b] == 1;
    for (int h = warp; h < G; h += S::kWarps) {
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
      const int hq = x.h * G + h;
      const float lse2 = (lt > 0.f) ? M + lg2(lt) : -INFINITY;
#pragma unroll
      for (int r = 0; r < D / 32; ++r) {
        const int d = lane + 32 * r;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < S::kWarps; ++w) o = fmaf(scratch[(w * G + h) * S::kSRow + d], wgt[w], o);
        o = (lt > 0.f) ? o / lt : 0.f;
        if (single)
          p.out[((size_t)x.b * p.H_q + hq) * D + d] = __float2bfloat16_rn(o);
        else
          p.o_part[((size_t)x.slot * p.H_q + hq) * D + d] = o;
      }
      if (lane == 0) {
        if (single)
          p.lse[(size_t)x.b * p.H_q + hq] = (lt > 0.f) ? lse2 * kLn2 : -INFINITY;
        else
          p.lse_part[(size_t)x.slot * p.H_q + hq] = lse2;
      }
    }
    // Leave together: the OR over all consumer threads of the abort flag is
    // the same value in every warp, so no warp waits alone at a barrier.
    if (named_bar_or(1, S::kWarps * 32, *abort_flag != 0)) return;
  }
}

template <int G, int D>
__global__ void __maxnreg__(kFmaMaxRegs)
    split_fma_kernel(Launch p) {
  using S = FmaShape<G, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* scratch = reinterpret_cast<float*>(smem + S::kStages * S::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
  uint64_t* empty = full + S::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S::kStages);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), S::kWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int n_units = p.hdr[kHdrNWork] * p.H_kv;
  if ((threadIdx.x >> 5) == S::kWarps)
    producer<G, D>(p, stages, full, empty, abort_flag, n_units);
  else
    consumer<G, D>(p, stages, scratch, full, empty, abort_flag, n_units);
}

template <int G, int D>
cudaError_t launch_one(const Launch& p, int grid, cudaStream_t stream) {
  using S = FmaShape<G, D>;
  static const cudaError_t attr = cudaFuncSetAttribute(
      split_fma_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (attr != cudaSuccess) return attr;
  split_fma_kernel<G, D><<<grid, S::kThreads, S::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int G, int D>
int ctas_one() {
  using S = FmaShape<G, D>;
  static int n = [] {
    cudaFuncSetAttribute(split_fma_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         S::kSmemBytes);
    int c = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, split_fma_kernel<G, D>, S::kThreads,
                                                      S::kSmemBytes) != cudaSuccess)
      c = 1;
    return c < 1 ? 1 : c;
  }();
  return n;
}

}  // namespace

bool fma_supported(int G, int D) {
  // G * D <= 512 keeps a lane's query and accumulator registers at <= 64 each.
  return (G == 1 || G == 2 || G == 4 || G == 8) && (D == 64 || D == 128) && G * D <= 512;
}

cudaError_t launch_split_fma(const Launch& p, int grid, cudaStream_t stream) {
  const int G = p.H_q / p.H_kv, D = p.D_qk;
  if (G == 1 && D == 64) return launch_one<1, 64>(p, grid, stream);
  if (G == 2 && D == 64) return launch_one<2, 64>(p, grid, stream);
  if (G == 4 && D == 64) return launch_one<4, 64>(p, grid, stream);
  if (G == 8 && D == 64) return launch_one<8, 64>(p, grid, stream);
  if (G == 1 && D == 128) return launch_one<1, 128>(p, grid, stream);
  if (G == 2 && D == 128) return launch_one<2, 128>(p, grid, stream);
  if (G == 4 && D == 128) return launch_one<4, 128>(p, grid, stream);
  return cudaErrorInvalidValue;
}

int fma_ctas_per_sm(int G, int D) {
  if (G == 1 && D == 64) return ctas_one<1, 64>();
  if (G == 2 && D == 64) return ctas_one<2, 64>();
  if (G == 4 && D == 64) return ctas_one<4, 64>();
  if (G == 8 && D == 64) return ctas_one<8, 64>();
  if (G == 1 && D == 128) return ctas_one<1, 128>();
  if (G == 2 && D == 128) return ctas_one<2, 128>();
  if (G == 4 && D == 128) return ctas_one<4, 128>();
  return 1;
}

}  // namespace da
