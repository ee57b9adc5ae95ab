// C ABI of the decode attention library: argument checks, workspace layout,
// plan construction and kernel launches.  Allocates nothing; synchronises the
// host only in the two documented read-back calls.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "merge.cuh"

namespace da {
bool mla_supported(int H_q);
}

namespace {

using namespace da;

struct Variant {
  int id, tile, min_tps, max_splits;
};

struct WsLayout {
  size_t n_splits, split_begin, work, item_desc, lse_part, o_part, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int check_problem(const da_problem* p) {
  if (!p) return DA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->num_q_heads < 1 || p->num_kv_heads < 1) return DA_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads) return DA_ERR_INVALID_ARG;
  if (p->head_dim_qk < 1 || p->head_dim_v < 1) return DA_ERR_INVALID_ARG;
  if (p->layout < DA_KV_CONTIGUOUS || p->layout > DA_KV_INDEXED) return DA_ERR_INVALID_ARG;
  if (p->layout == DA_KV_PAGED && p->page_size < 1) return DA_ERR_INVALID_ARG;
  if (p->width < 0) return DA_ERR_INVALID_ARG;
  if (p->layout != DA_KV_CONTIGUOUS && p->num_blocks < 0) return DA_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return DA_ERR_INVALID_ARG;
  if ((p->flags & ~DA_FLAG_TEST_STALL) != 0) return DA_ERR_INVALID_ARG;
  if (p->shared_latent != 0 && p->shared_latent != 1) return DA_ERR_INVALID_ARG;
  if (p->shared_latent && p->head_dim_v > p->head_dim_qk) return DA_ERR_INVALID_ARG;
  if (p->extra_width < 0 || p->extra_num_blocks < 0) return DA_ERR_INVALID_ARG;
  if (row_capacity(p->layout, p->width, p->page_size) + p->extra_width > 0x7fffffffLL)
    return DA_ERR_INVALID_ARG;
  if (p->kv_dtype != DA_KV_BF16 && p->kv_dtype != DA_KV_FP8_E4M3 && p->kv_dtype != DA_KV_NVFP4)
    return DA_ERR_INVALID_ARG;
  if (p->kv_dtype != DA_KV_BF16 &&
      !(std::isfinite(p->k_scale) && p->k_scale > 0.f && std::isfinite(p->v_scale) &&
        p->v_scale > 0.f))
    return DA_ERR_INVALID_ARG;
  return DA_OK;
}

// The kernel variant follows from the head configuration alone -- never from
// the batch size or the lengths.
int select_variant(const da_problem* p, Variant* v) {
  // quantized caches: one KV source; a shared latent cache in E4M3 only
  if (p->kv_dtype != DA_KV_BF16 &&
      (p->extra_width > 0 || (p->shared_latent && p->kv_dtype != DA_KV_FP8_E4M3)))
    return DA_ERR_UNSUPPORTED;
  if (p->shared_latent) {
    if (p->head_dim_qk == 576 && p->head_dim_v == 512 && p->num_kv_heads == 1 &&
        mla_supported(p->num_q_heads)) {
      *v = {DA_VARIANT_MLA, kMlaTile, kMlaMinTilesPerSplit, kMlaMaxSplits};
      return DA_OK;
    }
    return DA_ERR_UNSUPPORTED;
  }
  const int G = p->num_q_heads / p->num_kv_heads;
  // groups of at least 16 heads over a bf16, E4M3 or NVFP4 cache (NVFP4: an
  // even number of KV heads) with one source: the multi-head contractions go
  // to the tensor cores
  const bool tc_cache = p->kv_dtype == DA_KV_BF16 || p->kv_dtype == DA_KV_FP8_E4M3 ||
                        (p->kv_dtype == DA_KV_NVFP4 && p->num_kv_heads % 2 == 0);
  if (p->head_dim_qk == p->head_dim_v && tc_cache && p->extra_width == 0 &&
      gqa_tc_supported(G, p->head_dim_qk)) {
    *v = {DA_VARIANT_GQA_TC, kTcTile, kTcMinTilesPerSplit, kTcMaxSplits};
    return DA_OK;
  }
  if (p->head_dim_qk == p->head_dim_v && fma_supported(G, p->head_dim_qk)) {
    *v = {DA_VARIANT_FMA, kFmaTile, kFmaMinTilesPerSplit, kFmaMaxSplits};
    return DA_OK;
  }
  return DA_ERR_UNSUPPORTED;
}

bool layout_fits(const da_problem* p, int max_splits) {
  // work-list entries b * max_splits + s must fit in int32
  return (long long)p->batch * (max_splits + 1) < 0x7fffffffLL;
}

WsLayout ws_layout(const da_problem* p, int max_splits) {
  const size_t B = (size_t)p->batch, ms = (size_t)max_splits;
  const size_t Hq = (size_t)p->num_q_heads, Dv = (size_t)p->head_dim_v;
  WsLayout L;
  size_t off = kHdrBytes;
  L.n_splits = off;
  off = align256(off + 4 * B);
  L.split_begin = off;
  off = align256(off + 4 * B * (ms + 1));
  L.work = off;
  off = align256(off + 4 * B * ms);
  L.item_desc = off;
  off = align256(off + 16 * B * ms);
  L.lse_part = off;
  off = align256(off + 4 * B * ms * Hq);
  L.o_part = off;
  off = align256(off + 4 * B * ms * Hq * Dv);
  L.total = off;
  return L;
}

int sm_count(int dev) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

Launch make_launch(const da_plan* plan) {
  const da_problem& pr = plan->prob;
  uint8_t* ws = static_cast<uint8_t*>(plan->ws);
  Launch L;
  std::memset(&L, 0, sizeof(L));
  L.hdr = reinterpret_cast<int32_t*>(ws);
  L.n_splits = reinterpret_cast<const int32_t*>(ws + plan->off_n_splits);
  L.split_begin = reinterpret_cast<const int32_t*>(ws + plan->off_split_begin);
  L.work = reinterpret_cast<const int32_t*>(ws + plan->off_work);
  L.item_desc = reinterpret_cast<const int32_t*>(ws + plan->off_item_desc);
  L.lse_part = reinterpret_cast<float*>(ws + plan->off_lse_part);
  L.o_part = reinterpret_cast<float*>(ws + plan->off_o_part);
  L.num_blocks = pr.num_blocks;
  L.B = pr.batch;
  L.H_q = pr.num_q_heads;
  L.H_kv = pr.num_kv_heads;
  L.D_qk = pr.head_dim_qk;
  L.D_v = pr.head_dim_v;
  L.layout = pr.layout;
  L.page_size = pr.page_size;
  L.width = pr.width;
  L.capacity = (int)row_capacity(pr.layout, pr.width, pr.page_size);
  L.page_shift = -1;
  if (pr.layout == DA_KV_PAGED && pr.page_size > 0 && (pr.page_size & (pr.page_size - 1)) == 0) {
    int sh = 0;
    while ((1 << sh) < pr.page_size) ++sh;
    L.page_shift = sh;
  }
  L.max_splits = plan->max_splits;
  L.o_part_mla = plan->variant == DA_VARIANT_MLA;
  L.test_stall = (pr.flags & DA_FLAG_TEST_STALL) != 0;
  L.scale_log2 = pr.scale * kLog2e;
  if (pr.kv_dtype != DA_KV_BF16) {  // scores of scaled keys: scale * k_scale
    L.kv_type = pr.kv_dtype;
    L.scale_log2 *= pr.k_scale;
    L.v_scale = pr.v_scale;
    L.kv_rows = (pr.layout == DA_KV_CONTIGUOUS) ? (long long)pr.batch * pr.width
                : (pr.layout == DA_KV_PAGED)    ? pr.num_blocks * pr.page_size
                                                : pr.num_blocks;
  }
  return L;
}

// The most splits any row of `plan` can have: under INVARIANT a row of L
// entries has ceil(tiles / tps) splits with tps >= min_tiles_per_split and
// tiles <= ceil(capacity / tile), so n <= ceil(that / min_tiles_per_split);
// BALANCED may cut any row into max_splits.
int split_bound(const da_plan* plan) {
  if (plan->policy != DA_POLICY_INVARIANT) return plan->max_splits;
  const da_problem& pr = plan->prob;
  long long cap = row_capacity(pr.layout, pr.width, pr.page_size);
  if (plan->has_extra) cap += pr.extra_width;
  const long long tiles = (cap + plan->tile_tokens - 1) / plan->tile_tokens;
  const long long n = (tiles + plan->min_tiles_per_split - 1) / plan->min_tiles_per_split;
  return (int)std::min<long long>(std::max<long long>(n, 1), plan->max_splits);
}

int check_plan(const da_plan* plan) {
  if (!plan) return DA_ERR_INVALID_ARG;
  int rc = check_problem(&plan->prob);
  if (rc != DA_OK) return rc;
  Variant v;
  rc = select_variant(&plan->prob, &v);
  if (rc != DA_OK) return rc;
  if (plan->variant != v.id || plan->max_splits != v.max_splits) return DA_ERR_INVALID_ARG;
  if (plan->prob.batch > 0) {
    if (!plan->ws || !aligned(plan->ws, 256)) return DA_ERR_WORKSPACE;
    if (plan->ws_bytes < ws_layout(&plan->prob, v.max_splits).total) return DA_ERR_WORKSPACE;
  }
  return DA_OK;
}

}  // namespace

extern "C" {

const char* decode_attn_version(void) {
  static char buf[256];
  static std::once_flag once;
  std::call_once(once, [] {
    std::snprintf(buf, sizeof(buf),
                  "decode_attn 0.2 sm_103a; fma: tile=%d min_tiles=%d max_splits=%d; "
                  "mla: tile=%d min_tiles=%d max_splits=%d; "
                  "gqa_tc: tile=%d min_tiles=%d max_splits=%d; balanced fixed_overhead=%d",
                  kFmaTile, kFmaMinTilesPerSplit, kFmaMaxSplits, kMlaTile, kMlaMinTilesPerSplit,
                  kMlaMaxSplits, kTcTile, kTcMinTilesPerSplit, kTcMaxSplits,
                  kBalancedFixedOverhead);
  });
  return buf;
}

const char* decode_attn_status_string(int status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported head configuration";
    case DA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int decode_attn_split_constants(const da_problem* prob, int32_t* variant, int32_t* tile_tokens,
                                int32_t* min_tiles_per_split, int32_t* max_splits) {
  int rc = check_problem(prob);
  if (rc != DA_OK) return rc;
  Variant v;
  rc = select_variant(prob, &v);
  if (rc != DA_OK) return rc;
  if (variant) *variant = v.id;
  if (tile_tokens) *tile_tokens = v.tile;
  if (min_tiles_per_split) *min_tiles_per_split = v.min_tps;
  if (max_splits) *max_splits = v.max_splits;
  return DA_OK;
}

int decode_attn_workspace_bytes(const da_problem* prob, size_t* bytes) {
  int rc = check_problem(prob);
  if (rc != DA_OK) return rc;
  if (!bytes) return DA_ERR_INVALID_ARG;
  Variant v;
  rc = select_variant(prob, &v);
  if (rc != DA_OK) return rc;
  if (!layout_fits(prob, v.max_splits)) return DA_ERR_INVALID_ARG;
  *bytes = ws_layout(prob, v.max_splits).total;
  return DA_OK;
}

static int plan_impl(const da_problem* prob, int32_t policy, const int32_t* d_lengths,
                     const int32_t* d_extra_lengths, void* d_ws, size_t ws_bytes, da_plan* plan,
                     void* stream) {
  int rc = check_problem(prob);
  if (rc != DA_OK) return rc;
  if (!plan || (policy != DA_POLICY_INVARIANT && policy != DA_POLICY_BALANCED))
    return DA_ERR_INVALID_ARG;
  Variant v;
  rc = select_variant(prob, &v);
  if (rc != DA_OK) return rc;
  if (!layout_fits(prob, v.max_splits)) return DA_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(prob, v.max_splits);
  if (prob->batch > 0) {
    if (!d_lengths) return DA_ERR_INVALID_ARG;
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < L.total) return DA_ERR_WORKSPACE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms <= 0) return DA_ERR_CUDA;
  // CTAs that one (row, split) item occupies: one per KV head and head chunk
  // (CUDA-core variant), one per KV head (GQA tensor-core variant) or two, one
  // per half of D_v (shared-latent tensor-core variant).
  int gc = 1, chunks = 1;
  if (v.id == DA_VARIANT_FMA)
    fma_chunk_shape(prob->num_q_heads / prob->num_kv_heads, prob->head_dim_qk, &gc, &chunks);
  const int per_item = (v.id == DA_VARIANT_MLA) ? 2 : prob->num_kv_heads * chunks;
  // persistent CTAs: as many as can be resident at once (whole pairs for the
  // shared-latent variant)
  const long long slots =
      (v.id == DA_VARIANT_MLA)      ? (long long)mla_resident_ctas(sms)
      : (v.id == DA_VARIANT_GQA_TC) ? (long long)gqa_tc_resident_ctas(sms)
                                    : (long long)sms * fma_ctas_per_sm(prob->num_q_heads /
                                                                           prob->num_kv_heads,
                                                                       prob->head_dim_qk);
  const long long max_units = (long long)prob->batch * v.max_splits * per_item;

  da_plan P;
  std::memset(&P, 0, sizeof(P));
  P.prob = *prob;
  P.policy = policy;
  P.variant = v.id;
  P.tile_tokens = v.tile;
  P.min_tiles_per_split = v.min_tps;
  P.max_splits = v.max_splits;
  P.num_parts = (int)(slots / per_item > 0 ? kBalancedPartsPerSlot * (slots / per_item) : 1);
  P.fixed_overhead = kBalancedFixedOverhead;
  P.grid = (int)(max_units < slots ? (max_units > 0 ? max_units : 1) : slots);
  P.device = dev;
  P.has_extra = d_extra_lengths != nullptr;
  P.ws = d_ws;
  P.ws_bytes = ws_bytes;
  P.off_n_splits = L.n_splits;
  P.off_split_begin = L.split_begin;
  P.off_work = L.work;
  P.off_item_desc = L.item_desc;
  P.off_lse_part = L.lse_part;
  P.off_o_part = L.o_part;
  *plan = P;
  if (prob->batch == 0) return DA_OK;

  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  PlanLaunch pl;
  pl.lengths = d_lengths;
  pl.extra_lengths = d_extra_lengths;
  pl.extra_capacity = prob->extra_width;
  pl.hdr = reinterpret_cast<int32_t*>(ws);
  pl.n_splits = reinterpret_cast<int32_t*>(ws + L.n_splits);
  pl.split_begin = reinterpret_cast<int32_t*>(ws + L.split_begin);
  pl.work = reinterpret_cast<int32_t*>(ws + L.work);
  pl.item_desc = reinterpret_cast<int32_t*>(ws + L.item_desc);
  pl.B = prob->batch;
  pl.tile = v.tile;
  pl.min_tps = v.min_tps;
  pl.max_splits = v.max_splits;
  pl.capacity = (int)row_capacity(prob->layout, prob->width, prob->page_size);
  pl.policy = policy;
  pl.num_parts = P.num_parts;
  pl.fixed_overhead = P.fixed_overhead;
  if (launch_plan(pl, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

int decode_attn_plan(const da_problem* prob, int32_t policy, const int32_t* d_lengths,
                     void* d_ws, size_t ws_bytes, da_plan* plan, void* stream) {
  return plan_impl(prob, policy, d_lengths, nullptr, d_ws, ws_bytes, plan, stream);
}

int decode_attn_plan_extra(const da_problem* prob, int32_t policy, const int32_t* d_lengths,
                           const int32_t* d_extra_lengths, void* d_ws, size_t ws_bytes,
                           da_plan* plan, void* stream) {
  if (!prob || prob->extra_width < 1) return DA_ERR_INVALID_ARG;
  if (prob->batch > 0 && !d_extra_lengths) return DA_ERR_INVALID_ARG;
  static const int32_t dummy = 0;  // B = 0: any non-null marker will do
  return plan_impl(prob, policy, d_lengths, prob->batch > 0 ? d_extra_lengths : &dummy, d_ws,
                   ws_bytes, plan, stream);
}

static int run_impl(const da_plan* plan, const void* q, const void* k, const void* v,
                    const int32_t* table, const int32_t* lengths, const void* extra_k,
                    const void* extra_v, const int32_t* extra_indices,
                    const int32_t* extra_lengths, void* out, float* lse, void* stream) {
  int rc = check_plan(plan);
  if (rc != DA_OK) return rc;
  const da_problem& pr = plan->prob;
  if ((extra_k != nullptr) != (plan->has_extra != 0)) return DA_ERR_INVALID_ARG;
  if (pr.batch == 0) return DA_OK;
  if (extra_k) {
    if (!extra_indices || !extra_lengths || (!pr.shared_latent && !extra_v))
      return DA_ERR_INVALID_ARG;
    if (!aligned(extra_k, 16) || (extra_v && !aligned(extra_v, 16)) ||
        !aligned(extra_indices, 4) || !aligned(extra_lengths, 4))
      return DA_ERR_INVALID_ARG;
  }
  if (!q || !k || !lengths || !out || !lse) return DA_ERR_INVALID_ARG;
  if (!pr.shared_latent && !v) return DA_ERR_INVALID_ARG;
  if (pr.layout != DA_KV_CONTIGUOUS && !table) return DA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || (v && !aligned(v, 16)) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(lengths, 4) || (table && !aligned(table, 4)))
    return DA_ERR_INVALID_ARG;
  Launch L = make_launch(plan);
  L.q = static_cast<const __nv_bfloat16*>(q);
  L.k = static_cast<const __nv_bfloat16*>(k);
  L.v = static_cast<const __nv_bfloat16*>(pr.shared_latent ? k : v);
  L.table = table;
  L.lengths = lengths;
  L.out = static_cast<__nv_bfloat16*>(out);
  L.lse = lse;
  if (extra_k) {
    L.extra_k = static_cast<const __nv_bfloat16*>(extra_k);
    L.extra_v = static_cast<const __nv_bfloat16*>(pr.shared_latent ? extra_k : extra_v);
    L.extra_table = extra_indices;
    L.extra_lengths = extra_lengths;
    L.extra_num_blocks = pr.extra_num_blocks;
    L.extra_width = pr.extra_width;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = (plan->variant == DA_VARIANT_MLA)      ? launch_split_mla(L, plan->grid, s)
                        : (plan->variant == DA_VARIANT_GQA_TC) ? launch_split_gqa_tc(L, plan->grid, s)
                                                          : launch_split_fma(L, plan->grid, s);
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int decode_attn_run(const da_plan* plan, const void* q, const void* k, const void* v,
                    const int32_t* table, const int32_t* lengths, void* out, float* lse,
                    void* stream) {
  return run_impl(plan, q, k, v, table, lengths, nullptr, nullptr, nullptr, nullptr, out, lse,
                  stream);
}

int decode_attn_run_extra(const da_plan* plan, const void* q, const void* k, const void* v,
                          const int32_t* table, const int32_t* lengths, const void* extra_k,
                          const void* extra_v, const int32_t* extra_indices,
                          const int32_t* extra_lengths, void* out, float* lse, void* stream) {
  if (!extra_k) return DA_ERR_INVALID_ARG;
  return run_impl(plan, q, k, v, table, lengths, extra_k, extra_v, extra_indices, extra_lengths,
                  out, lse, stream);
}

int decode_attn_combine(const da_plan* plan, void* out, float* lse, void* stream) {
  int rc = check_plan(plan);
  if (rc != DA_OK) return rc;
  if (plan->prob.batch == 0) return DA_OK;
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) return DA_ERR_INVALID_ARG;
  Launch L = make_launch(plan);
  L.out = static_cast<__nv_bfloat16*>(out);
  L.lse = lse;
  return launch_combine(L, split_bound(plan), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_CUDA;
}

int decode_attn_forward(const da_problem* prob, int32_t policy, const void* q, const void* k,
                        const void* v, const int32_t* table, const int32_t* lengths,
                        void* d_ws, size_t ws_bytes, void* out, float* lse, void* stream) {
  da_plan plan;
  int rc = decode_attn_plan(prob, policy, lengths, d_ws, ws_bytes, &plan, stream);
  if (rc != DA_OK) return rc;
  rc = decode_attn_run(&plan, q, k, v, table, lengths, out, lse, stream);
  if (rc != DA_OK) return rc;
  return decode_attn_combine(&plan, out, lse, stream);
}

int decode_attn_forward_extra(const da_problem* prob, int32_t policy, const void* q,
                              const void* k, const void* v, const int32_t* table,
                              const int32_t* lengths, const void* extra_k, const void* extra_v,
                              const int32_t* extra_indices, const int32_t* extra_lengths,
                              void* d_ws, size_t ws_bytes, void* out, float* lse, void* stream) {
  da_plan plan;
  int rc = decode_attn_plan_extra(prob, policy, lengths, extra_lengths, d_ws, ws_bytes, &plan,
                                  stream);
  if (rc != DA_OK) return rc;
  rc = decode_attn_run_extra(&plan, q, k, v, table, lengths, extra_k, extra_v, extra_indices,
                             extra_lengths, out, lse, stream);
  if (rc != DA_OK) return rc;
  return decode_attn_combine(&plan, out, lse, stream);
}

int decode_attn_read_error(const da_plan* plan, int32_t* code, void* stream) {
  if (!plan || !code) return DA_ERR_INVALID_ARG;
  *code = 0;
  if (plan->prob.batch == 0) return DA_OK;
  if (!plan->ws) return DA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(code, static_cast<const int32_t*>(plan->ws) + kHdrError, sizeof(int32_t),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DA_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int decode_attn_copy_plan(const da_plan* plan, int32_t* n_splits, int32_t* split_begin,
                          int32_t* n_work, int32_t* work, void* stream) {
  if (!plan) return DA_ERR_INVALID_ARG;
  const size_t B = (size_t)plan->prob.batch, ms = (size_t)plan->max_splits;
  if (B == 0) {
    if (n_work) *n_work = 0;
    return DA_OK;
  }
  if (!plan->ws) return DA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(plan->ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n_splits && e == cudaSuccess)
    e = cudaMemcpyAsync(n_splits, ws + plan->off_n_splits, 4 * B, cudaMemcpyDeviceToHost, s);
  if (split_begin && e == cudaSuccess)
    e = cudaMemcpyAsync(split_begin, ws + plan->off_split_begin, 4 * B * (ms + 1),
                        cudaMemcpyDeviceToHost, s);
  if (n_work && e == cudaSuccess)
    e = cudaMemcpyAsync(n_work, reinterpret_cast<const int32_t*>(ws) + kHdrNWork, 4,
                        cudaMemcpyDeviceToHost, s);
  if (work && e == cudaSuccess)
    e = cudaMemcpyAsync(work, ws + plan->off_work, 4 * B * ms, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // extern "C"
