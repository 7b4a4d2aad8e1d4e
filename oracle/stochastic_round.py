"""Stochastic rounding to bf16, stated bit by bit.

TEST INFRASTRUCTURE ONLY; the product path never imports it.

Source: dew.training.optim, "stochastic_round_bf16": a value is rounded to
bf16 up or down with the probability of its distance to each; 16 uniform bits
are added below the kept mantissa of the fp32 pattern and the low half is
dropped, so the result rounds up exactly when the dropped bits plus the noise
carry; the noise is a counter-based hash of a seed and the element's flat
index; NaN stays NaN. "bf16_moments": the update runs on the moments widened
to fp32 and writes them back stochastically rounded, seeded by the step
count, the leaf and the moment.

Readings (the page names neither the hash nor how the seed is composed):
  * The hash is the 32-bit finaliser of MurmurHash3 (Austin Appleby, public
    domain), fmix32: x ^= x >> 16; x *= 0x85EBCA6B; x ^= x >> 13;
    x *= 0xC2B2AE35; x ^= x >> 16 (mod 2**32). It is cheap in 32-bit integer
    arithmetic, which the page's "a few integer ops per element" asks for.
  * key(seed, stream) = fmix32(fmix32(fmix32(stream) ^ seed_lo) ^ seed_hi),
    seed_lo / seed_hi the low and high 32 bits of the 64-bit seed. One hash
    serves two consecutive elements: the noise of flat element i is the low
    (i even) or high (i odd) 16 bits of fmix32(key + floor(i / 2) mod 2**32).
  * stream = 4 * (index of the tensor in its call) + moment, moment 0 for the
    Muon momentum or AdamW's first moment, 1 for AdamW's second moment, 2 for
    the parameter itself.
  * seed: AdamW uses its 1-based step count; Muon uses the per-step seed the
    caller passes.
  * The rule acts on the fp32 value (the update runs in fp32); the fp64
    oracle first rounds its value to the nearest fp32.
  * NaN becomes the quiet NaN of the same sign.
"""
from __future__ import annotations

import numpy as np

_M32 = 0xFFFFFFFF

MOMENT_FIRST = 0    # Muon momentum, AdamW exp_avg
MOMENT_SECOND = 1   # AdamW exp_avg_sq
MOMENT_PARAM = 2    # the parameter


def fmix32(x):
    """MurmurHash3's 32-bit finaliser, for a Python int or a uint32/uint64 array."""
    if isinstance(x, (int, np.integer)):
        x = int(x) & _M32
        x ^= x >> 16
        x = (x * 0x85EBCA6B) & _M32
        x ^= x >> 13
        x = (x * 0xC2B2AE35) & _M32
        return x ^ (x >> 16)
    x = np.asarray(x, dtype=np.uint64) & np.uint64(_M32)
    x ^= x >> np.uint64(16)
    x = (x * np.uint64(0x85EBCA6B)) & np.uint64(_M32)
    x ^= x >> np.uint64(13)
    x = (x * np.uint64(0xC2B2AE35)) & np.uint64(_M32)
    return x ^ (x >> np.uint64(16))


def sr_key(seed: int, stream: int) -> int:
    seed = int(seed) & ((1 << 64) - 1)
    return fmix32(fmix32(fmix32(int(stream) & _M32) ^ (seed & _M32)) ^ (seed >> 32))


def sr_stream(tensor_index: int, moment: int) -> int:
    return 4 * int(tensor_index) + int(moment)


def sr_noise16(key: int, index) -> np.ndarray:
    """16 uniform bits for each flat index (uint32 values in [0, 65536))."""
    idx = np.asarray(index, dtype=np.uint64)
    h = fmix32((np.uint64(key) + (idx >> np.uint64(1))) & np.uint64(_M32))
    shift = np.uint64(16) * (idx & np.uint64(1))
    return ((h >> shift) & np.uint64(0xFFFF)).astype(np.uint32)


def round_bf16_with_noise(x, noise16) -> np.ndarray:
    """The rounding rule with explicit noise: x (rounded to fp32 first, unless
    it is already a float32 array, whose bits are used as they are) plus 16
    noise bits below the kept mantissa, low half dropped. Returns the bf16
    values as float64."""
    x = np.asarray(x)
    if x.dtype != np.float32:
        x = x.astype(np.float64).astype(np.float32)
    f = np.ascontiguousarray(x)
    u = f.view(np.uint32).astype(np.uint64)
    r = np.asarray(noise16, dtype=np.uint64) & np.uint64(0xFFFF)
    hi = ((u + r) >> np.uint64(16)) & np.uint64(0xFFFF)
    nan = np.isnan(f)
    sign = (u >> np.uint64(31)) << np.uint64(15)
    hi = np.where(nan, sign | np.uint64(0x7FC0), hi)
    out = (hi << np.uint64(16)).astype(np.uint32).view(np.float32)
    return out.astype(np.float64)


def stochastic_round_bf16(x, seed: int, stream: int, index0: int = 0) -> np.ndarray:
    """bf16 values of x (any shape), element k drawing the noise of flat
    index index0 + k."""
    x = np.asarray(x, dtype=np.float64)
    idx = np.arange(index0, index0 + x.size, dtype=np.uint64)
    return round_bf16_with_noise(x.ravel(), sr_noise16(sr_key(seed, stream), idx)).reshape(x.shape)
