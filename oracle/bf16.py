"""Exact fp64 -> bf16 rounding (round to nearest, ties to even) and bf16 ULP.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

bf16 is IEEE binary32 with the low 16 fraction bits dropped: 1 sign bit,
8 exponent bits (bias 127), 7 stored fraction bits.  Rounding an fp64 value
straight to that format (rather than through fp32, which could round twice)
keeps the oracle's reference output exact.

FlashMLA issue #212 (Measurement) measures the batch-dependence it reports in
bf16 ULP: "1-2 ULP of bf16 near 1.0", max_absdiff 0.00195-0.0039.  ``ulp``
below states the unit those figures are in.
"""

from __future__ import annotations

import numpy as np

_MIN_NORMAL = 2.0 ** -126
_SUBNORMAL_QUANTUM = 2.0 ** -133  # spacing of bf16 subnormals
_MAX_FINITE = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_to_bf16(x):
    """Round fp64 values to the nearest bf16 value (ties to even); returns fp64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x)
    ax = np.abs(x)
    normal = finite & (ax >= _MIN_NORMAL)
    # Normal range: keep 8 significant bits.  The fp64 fraction has 52 bits,
    # bf16 keeps 7, so the rounding position is fraction bit 45.
    bits = x[normal].view(np.uint64)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bits = bits + np.uint64((1 << 44) - 1) + lsb
    bits &= ~np.uint64((1 << 45) - 1)
    out[normal] = bits.view(np.float64)
    # Subnormal range: a fixed quantum; np.round rounds half to even.
    sub = finite & (ax < _MIN_NORMAL)
    out[sub] = np.round(x[sub] / _SUBNORMAL_QUANTUM) * _SUBNORMAL_QUANTUM
    # Past the largest finite bf16 (after rounding) the value is infinite.
    over = finite & (np.abs(out) > _MAX_FINITE)
    out[over] = np.copysign(np.inf, x[over])
    return out


def ulp(x):
    """Spacing of bf16 values at |x| (the gap to the next larger bf16 magnitude)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, _MIN_NORMAL)))
    return np.exp2(e - 7)
