/*
 * decode_attn.h -- C ABI of the batch-invariant split-KV decode attention
 * library (GB300, sm_103a).
 *
 * What the library computes.  For every query row b and query head j, plain
 * softmax attention over the row's own KV list (FlashMLA issue #212, "Sparse
 * MLA decode is not batch-invariant", Summary and Measurement: the call
 * flash_mla_with_kvcache(q, indices, topk_length, ...) returning per-row
 * output and LSE):
 *
 *     s_i = scale * q[b, j, :] . K_b[i, h, :]        h = j / (H_q / H_kv)
 *     lse[b, j] = log sum_i exp(s_i)                 (natural log, fp32)
 *     out[b, j, :] = sum_i exp(s_i - lse) V_b[i, h, :] (bf16, round to nearest even)
 *
 * How.  A row's KV list is cut into tiles of T entries and the tiles into
 * splits (one unit of GPU work each).  Under DA_POLICY_INVARIANT the split
 * count and boundaries of a row depend only on its own length and compile-time
 * constants (same page, "Question": the opt-in mode whose split count derives
 * only from the row's own sequence length); every split's partial is merged
 * by an fp32 log-sum-exp combine in split order.  A row's output and LSE are
 * therefore bitwise identical whatever its batchmates and its position in the
 * batch.  DA_POLICY_BALANCED re-derives the batch-wide quota the same page
 * names as the cause ("Where it comes from": payload = ceil_div(total_num_
 * blocks, num_sm_parts) + fixed_overhead_num_blocks, then greedy packing); it
 * exists to measure what invariance costs and is NOT batch-invariant.
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses; the caller owns every
 *     buffer, including the workspace.  The library allocates no memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is only enqueued; no entry point synchronises the host
 *     except decode_attn_read_error and decode_attn_copy_plan.
 *   - Return value: DA_OK or a DA_ERR_* status; nothing is enqueued when the
 *     status is not DA_OK.  No entry point aborts, traps or prints.
 *   - bf16 tensors are raw IEEE bfloat16 bit patterns (uint16).
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------- */
#define DA_OK 0
#define DA_ERR_INVALID_ARG 1 /* null pointer, bad size, misaligned buffer  */
#define DA_ERR_UNSUPPORTED 2 /* head config / dims without a kernel        */
#define DA_ERR_WORKSPACE 3   /* workspace missing, misaligned or too small */
#define DA_ERR_CUDA 4        /* a CUDA runtime call or launch failed       */

/* ---- split policies ------------------------------------------------- */
#define DA_POLICY_INVARIANT 0 /* per-row split rule: batch-invariant        */
#define DA_POLICY_BALANCED 1  /* batch-wide quota: the counter-example      */

/* ---- KV cache layouts ----------------------------------------------- */
/* contiguous: k,v = [batch, width, H_kv, D]; entry t of row b = [b, t]     */
#define DA_KV_CONTIGUOUS 0
/* paged: k,v = [num_blocks, page_size, H_kv, D]; table = int32[batch,
 * width] of page ids; entry t of row b = [table[b, t / page_size],
 * t % page_size]                                                           */
#define DA_KV_PAGED 1
/* indexed (top-k gather): k,v = [num_blocks, H_kv, D]; table =
 * int32[batch, width] of slot indices; entry t of row b = [table[b, t]];
 * entries at t >= length are never read                                   */
#define DA_KV_INDEXED 2

/* ---- KV element types (da_problem.kv_dtype) ------------------------- */
#define DA_KV_BF16 0     /* bf16 K and V                                      */
/* One byte per element in the 8-bit E4M3 floating-point layout (bias 7,
 * subnormals, no infinities, S.1111.111 = NaN) with one fp32 scale per cache:
 * element value = scale * e4m3(byte).  The pages run low-precision
 * checkpoints (FlashMLA issue #212, Environment: NVFP4 DeepSeek-V4-Flash;
 * gllm issue #98, Observation: NVFP4 Nemotron) but name no cache format;
 * this is the library's reading.  The kernel converts each byte exactly to
 * fp32, applies k_scale to the softmax scale and v_scale to a unit's output
 * (fixed roundings, independent of the batch).  One KV source only
 * (DA_ERR_UNSUPPORTED otherwise).  DA_VARIANT_MLA for a shared latent cache
 * (576/512: scores from k_scale * the row's 576 bytes, values from v_scale *
 * its first 512), DA_VARIANT_GQA_TC for groups of 16 or more heads at
 * D = 128, else DA_VARIANT_FMA.                                            */
#define DA_KV_FP8_E4M3 1
/* NVFP4: each head's row of D elements is stored as D/2 bytes of 4-bit E2M1
 * codes (element 2j in the low nibble of byte j; magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6) and D/16 E4M3 block scales, one per 16 consecutive elements, with
 * one fp32 scale per cache: element value = scale * e4m3(block) * e2m1(code).
 * A cache buffer (k or v) holds all its codes first, laid out like a bf16
 * cache with D/2 bytes per head row ([rows, H_kv, D/2], rows = batch*width
 * contiguous, num_blocks*page_size paged, num_blocks indexed), and right
 * after them, at byte offset rows*H_kv*D/2, the block scales [rows, H_kv,
 * D/16] in the same order.  Same reading of the pages and the same rules as
 * DA_KV_FP8_E4M3 (k_scale, v_scale, one KV source; DA_VARIANT_GQA_TC only
 * when H_kv is even as well).  The kernel turns each code and each block
 * scale into f16 exactly and multiplies them in f16 (exact: at most six
 * significant bits).                                                       */
#define DA_KV_NVFP4 2

/* ---- kernel variants (chosen from the head config only, never B) ----- */
#define DA_VARIANT_FMA 0 /* CUDA-core fp32 FMA, H_q/H_kv in 1..128, D in {64,128}    */
/* tcgen05 tensor cores, shared latent 576/512, 16..128 heads (bf16, or E4M3
 * converted to f16 in shared memory with one KV source)                     */
#define DA_VARIANT_MLA 1
/* tcgen05 tensor cores, separate K and V (bf16, or E4M3 or NVFP4 converted
 * to f16 in shared memory; NVFP4 with an even H_kv), 16..128 query heads per
 * KV head, D = 128, one KV source (other configs of >= 16 heads:
 * DA_VARIANT_FMA)                                                           */
#define DA_VARIANT_GQA_TC 2

/* ---- device-detected input errors (decode_attn_read_error bits) ----- */
#define DA_DEVERR_LENGTH 1  /* a length < 0 or above capacity; it was clamped  */
#define DA_DEVERR_INDEX 2   /* a page id / slot index out of range; not read   */
#define DA_DEVERR_TIMEOUT 4 /* a pipeline wait hit its limit; kernel bailed out */

/* ---- da_problem.flags ------------------------------------------------ */
/* Test hook for the time-out path of the tensor-core variants, never for a
 * production call: with this flag the MMA-issuing thread of every CTA of
 * DA_VARIANT_MLA and DA_VARIANT_GQA_TC first waits on an mbarrier that
 * nothing signals, with a 2 ms limit.  That wait runs out, the kernel records
 * DA_DEVERR_TIMEOUT, every role leaves its loop, the copies in flight and the
 * tensor-core work are drained and tensor memory is freed before the CTA
 * exits, so the context stays usable; that call's outputs are unspecified.
 * The CUDA-core variant has no such waits and ignores the flag. */
#define DA_FLAG_TEST_STALL 1u

/* Problem description.  Plain data, filled by the caller. */
typedef struct da_problem {
  int32_t batch;         /* B >= 0 query rows                                 */
  int32_t num_q_heads;   /* H_q >= 1                                          */
  int32_t num_kv_heads;  /* H_kv >= 1, divides H_q                            */
  int32_t head_dim_qk;   /* D_qk: q and K row length                          */
  int32_t head_dim_v;    /* D_v: V row and output length                      */
  int32_t layout;        /* DA_KV_*                                           */
  int32_t page_size;     /* paged only: entries per page (>= 1)               */
  int32_t width;         /* contiguous: Lmax; paged: table row width (pages); */
                         /* indexed: index row width (max top-k)              */
  int64_t num_blocks;    /* paged: pages in the cache; indexed: slots;        */
                         /* contiguous: ignored                               */
  float scale;           /* softmax scale, applied in fp32 to the fp32 dot    */
  int32_t shared_latent; /* 1: one latent cache, v == NULL, V = K[..., :D_v]  */
  uint32_t flags;        /* 0, or DA_FLAG_TEST_STALL (tests only)             */
  /* Optional second KV source (the *_extra entry points): an index-gathered */
  /* cache [extra_num_blocks, H_kv, D] whose entries continue each row's     */
  /* list after its main entries.  0 / 0 when unused.                         */
  int32_t extra_width;      /* extra index row width (max extra entries)      */
  int64_t extra_num_blocks; /* slots in the extra cache                       */
  int32_t kv_dtype;         /* DA_KV_BF16 (0), DA_KV_FP8_E4M3, DA_KV_NVFP4    */
  float k_scale;            /* quantized caches: K scale (finite, > 0)        */
  float v_scale;            /* quantized caches: V scale (finite, > 0)        */
} da_problem;

/* A plan: filled by decode_attn_plan, read by run/combine.  Host memory,
 * owned by the caller; its fields are informative and must not be edited.
 * It stays valid while the workspace and the lengths it was built from are
 * unchanged (rebuild it every decode step, like the page's fresh
 * FlashMLASchedMeta). */
typedef struct da_plan {
  da_problem prob;
  int32_t policy;              /* DA_POLICY_*                                  */
  int32_t variant;             /* DA_VARIANT_*                                 */
  int32_t tile_tokens;         /* T: KV entries per tile                       */
  int32_t min_tiles_per_split; /* INVARIANT rule constant                      */
  int32_t max_splits;          /* splits per row at most; also the slot stride */
  int32_t num_parts;           /* BALANCED: parts the quota divides into       */
  int32_t fixed_overhead;      /* BALANCED: tiles charged per split            */
  int32_t grid;                /* persistent CTAs decode_attn_run launches     */
  int32_t device;              /* CUDA device the plan was made on             */
  int32_t has_extra;           /* 1: built by decode_attn_plan_extra           */
  void* ws;                    /* the workspace given to decode_attn_plan      */
  size_t ws_bytes;
  uint64_t off_n_splits;       /* int32[B]: splits of row b                    */
  uint64_t off_split_begin;    /* int32[B][max_splits+1]: boundaries, tiles    */
  uint64_t off_work;           /* int32[B*max_splits]: b*max_splits + s list   */
  uint64_t off_item_desc;      /* int32[B*max_splits][4]: per work item        */
                               /* {slot (~slot if the row has one split),      */
                               /*  first tile, end tile, clamped length}       */
  uint64_t off_lse_part;       /* float[B*max_splits][H_q]: split LSE (log2)   */
  uint64_t off_o_part;         /* float[B*max_splits][H_q][D_v]: split output  */
} da_plan;

/* Library version and the compile-time split constants, as text. */
const char* decode_attn_version(void);

/* Human-readable name of a DA_* status code (static string). */
const char* decode_attn_status_string(int status);

/* The kernel variant and split constants `prob` would use.  Any output
 * pointer may be NULL.  Returns DA_ERR_UNSUPPORTED when no kernel exists for
 * the head config. */
int decode_attn_split_constants(const da_problem* prob, int32_t* variant,
                                int32_t* tile_tokens, int32_t* min_tiles_per_split,
                                int32_t* max_splits);

/* Workspace bytes decode_attn_plan/run/combine need for `prob` (either
 * policy).  The workspace must be device memory aligned to 256 bytes. */
int decode_attn_workspace_bytes(const da_problem* prob, size_t* bytes);

/* Build the split plan on the device.
 *   d_lengths: int32[B] device array of KV lengths (top-k length for the
 *              indexed layout).  Values < 0 or above the layout's capacity
 *              (contiguous: width; paged: width*page_size; indexed: width)
 *              are clamped and flagged DA_DEVERR_LENGTH.
 *   d_ws, ws_bytes: caller-owned device workspace (see workspace_bytes).
 *   plan: host struct, filled on return.
 * Enqueues one small kernel on `stream`; also resets the device error word. */
int decode_attn_plan(const da_problem* prob, int32_t policy, const int32_t* d_lengths,
                     void* d_ws, size_t ws_bytes, da_plan* plan, void* stream);

/* The split kernel: every (row, split, KV head) partial.
 *   q:       bf16 [B, H_q, D_qk], 16-byte aligned
 *   k, v:    caches in prob->layout of prob->kv_dtype (bf16, E4M3 bytes, or
 *            NVFP4 codes then block scales); v NULL when shared_latent;
 *            16-byte aligned
 *   table:   int32 [B, width] page ids / slot indices (NULL for contiguous)
 *   lengths: the same int32[B] device array given to decode_attn_plan
 *   out:     bf16 [B, H_q, D_v]; lse: float [B, H_q] (natural log)
 * Rows with a single split are written final here; the other rows' partials
 * go to the workspace for decode_attn_combine.  Out-of-range page ids or
 * indices are not dereferenced: they set DA_DEVERR_INDEX and leave the
 * affected rows' outputs unspecified. */
int decode_attn_run(const da_plan* plan, const void* q, const void* k, const void* v,
                    const int32_t* table, const int32_t* lengths, void* out, float* lse,
                    void* stream);

/* Fixed-order fp32 LSE merge of the partials of every multi-split row into
 * out (bf16) and lse (float).  Must follow decode_attn_run on the same plan
 * (stream order is the only synchronisation). */
int decode_attn_combine(const da_plan* plan, void* out, float* lse, void* stream);

/* plan + run + combine in one call (same arguments, same results). */
int decode_attn_forward(const da_problem* prob, int32_t policy, const void* q, const void* k,
                        const void* v, const int32_t* table, const int32_t* lengths,
                        void* d_ws, size_t ws_bytes, void* out, float* lse, void* stream);

/* The forward pass without a caller-supplied workspace, for callers that
 * cannot allocate device memory (for example a plugin whose host process owns
 * every device allocation, or a latency-critical path that cannot afford the
 * synchronisation a cudaMalloc may bring).  The pages have no counterpart to
 * this entry point; it only changes where the scratch lives.
 *
 * Same arguments and results as decode_attn_forward minus the workspace.
 * The scratch is one file-scope device array of DA_STATIC_WORKSPACE_BYTES
 * (64 MiB) per device, held until the process exits from the time the
 * library's code is loaded on that device.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress, with that device
 * current) and caches it; make that first call before any stream capture.
 * The cached address is stale after cudaDeviceReset: do not call this entry
 * point again in a process that reset the device.  Nothing is allocated,
 * here or later.  A problem whose workspace (decode_attn_workspace_bytes)
 * exceeds DA_STATIC_WORKSPACE_BYTES is rejected with DA_ERR_WORKSPACE before
 * anything is enqueued.  All calls on a device share the one array and it
 * keeps the last call's contents (the plan rewrites everything a call reads,
 * including the error word), so calls whose work overlaps on the GPU --
 * different streams without ordering, or concurrent host threads -- race and
 * corrupt each other's results: serialise them.
 *
 * plan_out (host, may be NULL): on DA_OK, receives the call's plan, whose
 * workspace is the static array; decode_attn_read_error(plan_out, ...) then
 * reads the device input-check bits (DA_DEVERR_*) of this call, as long as no
 * later call of this entry point on the device has overwritten them. */
#define DA_STATIC_WORKSPACE_BYTES (64u << 20)
int decode_attn_forward_static(const da_problem* prob, int32_t policy, const void* q,
                               const void* k, const void* v, const int32_t* table,
                               const int32_t* lengths, void* out, float* lse, void* stream,
                               da_plan* plan_out);

/* The same three steps over two KV sources per row.  Row b attends over its
 * main list (as above) followed by extra_lengths[b] entries gathered from a
 * second cache: entry t of that part is extra_k[extra_indices[b, t]] (values
 * extra_v[...], or the leading D_v dims of extra_k when shared_latent).  This
 * is the sparse decode call of FlashMLA issue #212 with
 * extra_indices_in_kvcache / extra_topk_length (Measurement, item 2, and the
 * Environment's "sparse decode path with extra_k_cache").  The row's split
 * plan is the INVARIANT (or BALANCED) rule on its total length, so the extra
 * part changes nothing else: a row's bits still depend only on its own two
 * lists.  prob->extra_width and prob->extra_num_blocks describe the extra
 * cache; extra_indices is int32 [B, extra_width]; extra lengths beyond
 * extra_width are clamped and flagged DA_DEVERR_LENGTH, indices out of
 * [0, extra_num_blocks) flag DA_DEVERR_INDEX and are not read.  A plan made
 * by decode_attn_plan_extra must be run by decode_attn_run_extra (and the
 * other plans by decode_attn_run); anything else is DA_ERR_INVALID_ARG. */
int decode_attn_plan_extra(const da_problem* prob, int32_t policy, const int32_t* d_lengths,
                           const int32_t* d_extra_lengths, void* d_ws, size_t ws_bytes,
                           da_plan* plan, void* stream);
int decode_attn_run_extra(const da_plan* plan, const void* q, const void* k, const void* v,
                          const int32_t* table, const int32_t* lengths, const void* extra_k,
                          const void* extra_v, const int32_t* extra_indices,
                          const int32_t* extra_lengths, void* out, float* lse, void* stream);
int decode_attn_forward_extra(const da_problem* prob, int32_t policy, const void* q,
                              const void* k, const void* v, const int32_t* table,
                              const int32_t* lengths, const void* extra_k, const void* extra_v,
                              const int32_t* extra_indices, const int32_t* extra_lengths,
                              void* d_ws, size_t ws_bytes, void* out, float* lse, void* stream);

/* Synchronise `stream`, then read the device error word (DA_DEVERR_* bits)
 * written since the last decode_attn_plan on this workspace. */
int decode_attn_read_error(const da_plan* plan, int32_t* code, void* stream);

/* Synchronise `stream`, then copy the plan's device arrays to host memory
 * (any pointer may be NULL): n_splits int32[B], split_begin
 * int32[B*(max_splits+1)], *n_work, work int32[B*max_splits]. */
int decode_attn_copy_plan(const da_plan* plan, int32_t* n_splits, int32_t* split_begin,
                          int32_t* n_work, int32_t* work, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
