"""FP8 E4M3 key/value cache entries decoded exactly to fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages run low-precision checkpoints -- "Sparse MLA decode is not
batch-invariant" (FlashMLA issue #212, Environment) an NVFP4 DeepSeek-V4-Flash
on the sparse decode path, "Greedy outputs depend on batch composition" (gllm
issue #98, Observation) an NVFP4 Nemotron -- but name no KV cache format.
The reading used here and by the library: a quantized cache holds one byte
per K or V element in the E4M3 layout of the 8-bit floating-point formats
shared by current GPUs (1 sign bit, 4 exponent bits with bias 7, 3 fraction
bits, subnormals at exponent field 0, no infinities, the two codes S.1111.111
meaning NaN), and one fp32 scale per cache multiplies every decoded element:

    value = scale * (-1)^s * 2^(e - 7) * (1 + f / 8)     for e = 1 .. 15
    value = scale * (-1)^s * 2^(-6)    * (f / 8)         for e = 0

The attention over the decoded values is then ``attention.attend`` unchanged.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0  # largest finite magnitude: e = 15, f = 6


def decode_e4m3(codes):
    """fp64 values of E4M3 byte codes (any integer array of values 0..255)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    f = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(f / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def dequantize(codes, scale):
    """``scale * decode_e4m3(codes)`` in fp64 (the cache's real values)."""
    return decode_e4m3(codes) * np.float64(scale)
