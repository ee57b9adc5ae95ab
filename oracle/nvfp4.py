"""NVFP4 weight matrices decoded exactly to fp64, and the activation-rounded
matrix product they enter.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Greedy outputs depend on batch composition (NVFP4 GEMV/GEMM switch at 32
rows is a candidate)" (gllm issue #98, Candidate cause) describes a weight
matmul whose kernel is picked by the row count n: up to 32 rows a fused
dequantizing GEMV keeps the activations in f32, above that the weights are
unpacked to bf16 and a tensor-core GEMM runs on bf16-rounded activations.
The same page (Next steps) proposes making both paths round the activations
to bf16, so that the switch changes speed and not results.  What is computed
here is that agreed result, written as its plain definition:

    y[i, o] = sum_k bf16(x[i, k]) * W[o, k]

with every product and the sum exact (fp64; the inputs have few significant
bits, so fp64 loses nothing until the sum).

The page names the format (NVFP4) but not its layout.  The reading used here
and by the library:

* one E2M1 code per weight: sign bit 3, exponent bits 2..1 (bias 1),
  fraction bit 0; exponent 0 is the subnormal range, so the magnitudes are
  0, 0.5, 1, 1.5, 2, 3, 4, 6;
* two codes per byte along K, element 2j in the low nibble of byte j of the
  row, element 2j + 1 in the high nibble; ``codes`` is uint8 [N, K / 2];
* one E4M3 scale per 16 consecutive weights of a row (``scales`` uint8
  [N, K / 16], decoded by ``fp8.decode_e4m3``);
* one fp32 scale for the whole matrix;

    W[o, k] = global_scale * e4m3(scales[o, k // 16]) * e2m1(nibble(o, k)).
"""

from __future__ import annotations

import numpy as np

from . import bf16, fp8


def decode_e2m1(codes):
    """fp64 values of 4-bit E2M1 codes (integers 0..15)."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    normal = np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int64))
    subnormal = m / 2.0
    return sign * np.where(e == 0, subnormal, normal)


def unpack(codes):
    """uint8 [N, K / 2] -> E2M1 code integers [N, K] (low nibble first)."""
    c = np.asarray(codes).astype(np.int64)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = (c >> 4) & 0xF
    return out


def dequantize(codes, scales, global_scale):
    """The weight matrix W [N, K] in fp64."""
    vals = decode_e2m1(unpack(codes))
    s = fp8.decode_e4m3(scales)
    block = np.repeat(s, 16, axis=-1)
    if block.shape != vals.shape:
        raise ValueError(f"scales {np.shape(scales)} do not cover codes {np.shape(codes)}")
    return np.float64(global_scale) * block * vals


def dequantize_cache(codes, scales, global_scale):
    """A key or value cache stored as NVFP4, decoded to fp64.

    The pages' models are NVFP4 checkpoints ("Sparse MLA decode is not
    batch-invariant", Environment; "Greedy outputs depend on batch
    composition", Observation) but no page names a KV cache format.  The
    reading used here and by the library takes the weight layout above along
    a head's row: ``codes`` uint8 ``[..., H_kv, D / 2]`` (element 2j in the low
    nibble of byte j), ``scales`` uint8 ``[..., H_kv, D / 16]`` (one E4M3 scale
    per 16 consecutive elements of the row), one fp32 scale per cache:

        value[..., h, d] = global_scale * e4m3(scales[..., h, d // 16])
                           * e2m1(nibble d of row h)

    Returns fp64 ``[..., H_kv, D]``; ``attention.attend`` then runs unchanged.
    """
    return dequantize(codes, scales, global_scale)


def round_activations(x):
    """The agreed activation precision: fp32 values rounded to bf16 (RNE)."""
    return bf16.round_to_bf16(np.asarray(x, dtype=np.float64))


def matmul(x, codes, scales, global_scale):
    """y [n, N] = bf16(x) [n, K] @ W[N, K]^T in fp64."""
    xr = round_activations(x)
    w = dequantize(codes, scales, global_scale)
    return xr @ w.T


def abs_products(x, codes, scales, global_scale):
    """sum_k |bf16(x[i, k]) * W[o, k]| [n, N]: the magnitude that bounds the
    rounding error of any fp32 evaluation order of the sum."""
    xr = np.abs(round_activations(x))
    w = np.abs(dequantize(codes, scales, global_scale))
    return xr @ w.T
