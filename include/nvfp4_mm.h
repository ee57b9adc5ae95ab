/*
 * nvfp4_mm.h -- C ABI of the batch-invariant NVFP4 weight matmul (GB300,
 * sm_103a), built into the same shared library as decode_attn.h and sharing
 * its status codes (DA_OK, DA_ERR_*).
 *
 * Why it exists.  "Greedy outputs depend on batch composition (NVFP4
 * GEMV/GEMM switch at 32 rows is a candidate)" (gllm issue #98, Candidate
 * cause) traces batch-dependent greedy decoding to a weight matmul whose
 * kernel is chosen by the number of activation rows n: a dequantizing GEMV
 * with f32 activations up to 32 rows, a bf16 tensor-core GEMM above.  The
 * same page (Next steps) proposes one activation precision, bf16, for both,
 * so the switch changes speed and not results.  This library goes one step
 * further: one arithmetic for every n, so a row's result is bitwise the same
 * whatever else shares the call.
 *
 * What it computes.  For activations x [n, K] and an NVFP4 weight W [N, K]:
 *
 *     xr[i, k]  = bf16(x[i, k])                      round to nearest even
 *     W[o, k]   = e4m3(scales[o, k / 16]) * e2m1(nibble(o, k))   (exact in bf16)
 *     P_c[i, o] = sum over k in chunk c of xr[i, k] * W[o, k]
 *                 (fp32 accumulation on the tensor cores, K ascending in
 *                  steps of 16; chunk c = k in [c * 1024, (c + 1) * 1024))
 *     y[i, o]   = global_scale * (((P_0 + P_1) + P_2) + ...)      fp32
 *     y_bf16    = bf16(y)                            round to nearest even
 *
 * The chunking (NVFP4_MM_K_CHUNK) and the order of every sum depend only on
 * K, never on n, on the other rows or on where row i sits in x.
 *
 * Weight format (the page names NVFP4 but not its layout; this is the
 * reading):
 *   codes   uint8 [N, K / 2]  two E2M1 codes per byte along K, element 2j of
 *                             a row in the low nibble of byte j.  E2M1: sign
 *                             bit 3, exponent bits 2..1 (bias 1), fraction
 *                             bit 0; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *   scales  uint8 [N, K / 16] one E4M3 code (sign, 4 exponent bits with bias
 *                             7, 3 fraction bits; 0x7F / 0xFF are NaN) per 16
 *                             consecutive weights of a row.
 *   global_scale              one finite fp32 factor for the whole matrix.
 *
 * Conventions are those of decode_attn.h: device pointers owned by the
 * caller, `stream` a cudaStream_t passed as void*, no allocation, no host
 * synchronisation (except nvfp4_mm_read_error), DA_OK or a DA_ERR_* status
 * with nothing enqueued on error, no abort, trap or print.
 */
#ifndef NVFP4_MM_H
#define NVFP4_MM_H

#include <stddef.h>
#include <stdint.h>

#include "decode_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_MM_TILE_N 128   /* output features per tensor-core tile (MMA M) */
#define NVFP4_MM_ROW_TILE 32  /* activation rows per tile (MMA N)              */
#define NVFP4_MM_K_CHUNK 1024 /* K per partial sum P_c                         */

#define NVFP4_X_F32 0  /* activations given as fp32: rounded to bf16 on the device */
#define NVFP4_X_BF16 1 /* activations given as bf16: used as they are             */

/* Device workspace bytes for one call with n activation rows, N outputs and
 * reduction length K (0 when the shape is not supported).  It holds a 256-byte
 * header, one counter per output tile, the rounded activations (n rounded up
 * to NVFP4_MM_ROW_TILE rows) and, when K > NVFP4_MM_K_CHUNK, the fp32 partial
 * sums P_c.  Its contents need no initialisation. */
size_t nvfp4_mm_workspace_bytes(int32_t n, int32_t N, int32_t K);

/* y = global_scale * bf16(x) @ W^T as defined above.
 *   x       [n, K], fp32 (x_dtype NVFP4_X_F32) or bf16 (NVFP4_X_BF16),
 *           row-major, 16-byte aligned.
 *   codes   uint8 [N, K / 2], scales uint8 [N, K / 16], row-major; codes
 *           16-byte aligned, scales 4-byte aligned.
 *   y       fp32 [n, N], row-major, required.
 *   y_bf16  bf16 [n, N] or NULL; 8-byte aligned.
 *   ws      device workspace of at least nvfp4_mm_workspace_bytes(n, N, K)
 *           bytes, 256-byte aligned; reused by the next call only after this
 *           one's work on `stream` is ordered before it.
 * Supported shapes: n >= 0 (n = 0 enqueues nothing), N a positive multiple of
 * NVFP4_MM_TILE_N, K a positive multiple of 64; n * K and n * N below 2^31.
 * Errors: DA_ERR_INVALID_ARG (null or misaligned pointer, non-finite
 * global_scale, unknown x_dtype), DA_ERR_UNSUPPORTED (shape), DA_ERR_WORKSPACE,
 * DA_ERR_CUDA (a launch failed).  A pipeline wait inside the kernel that
 * hits its time limit records DA_DEVERR_TIMEOUT in the workspace header and
 * the kernel returns; y is then undefined. */
int nvfp4_mm(const void* x, int32_t x_dtype, const uint8_t* codes, const uint8_t* scales,
             float global_scale, int32_t n, int32_t N, int32_t K, float* y, void* y_bf16,
             void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then read the device error word (DA_DEVERR_* bits)
 * of the most recent nvfp4_mm call on workspace `ws` (each call clears it
 * when its first kernel starts; reading clears it too). */
int nvfp4_mm_read_error(void* ws, int32_t* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_MM_H */
