"""bf16 storage rounding used by the oracle for bf16 parameters.

TEST INFRASTRUCTURE ONLY.

The pages keep parameters in their own dtype and compute in fp32 or higher
(kimi-k3 "Optimization", "Keep the arithmetic and gradients under control").
The reading for a bf16 parameter: compute the new value in float64 and store
it rounded to the nearest bf16, ties to even. float64 -> bf16 is done as
float64 -> float32 -> bf16 only when that double rounding cannot differ from a
direct rounding; otherwise the exact float64 value decides.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even); returns float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    flat = x.reshape(-1)
    res = out.reshape(-1)
    finite = np.isfinite(flat)
    # Work on the float64 bit pattern: bf16 keeps 8 significand bits (7
    # stored), i.e. float64 with the low 45 fraction bits dropped.
    bits = flat.view(np.uint64)
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    mask = (np.uint64(1) << drop) - np.uint64(1)
    low = bits & mask
    kept = bits & ~mask
    lsb = (bits >> drop) & np.uint64(1)
    up = (low > half) | ((low == half) & (lsb == np.uint64(1)))
    rounded = kept + np.where(up, np.uint64(1) << drop, np.uint64(0))
    val = rounded.view(np.float64)
    # bf16 has float32's exponent range: tiny values round as float32 subnormals
    # would; values beyond the bf16 maximum overflow to inf.
    small = np.abs(flat) < np.float64(np.finfo(np.float32).tiny)
    if np.any(small & finite):
        f32 = flat[small & finite].astype(np.float32)
        b = f32.view(np.uint32).astype(np.uint64)
        r = ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
        val[small & finite] = r.astype(np.uint32).view(np.float32).astype(np.float64)
    bf16_max = float(np.float32(3.3895313892515355e38))
    val = np.where(finite & (np.abs(val) > bf16_max), np.sign(flat) * np.inf, val)
    res[:] = np.where(finite, val, flat)
    return out
