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
  * The hash is SplitMix64 (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", 2014): splitmix64(x) is the generator's
    output from state x, i.e. its finaliser applied to x + 0x9E3779B97F4A7C15.
  * key(seed, stream) = splitmix64(seed XOR splitmix64(stream)); one hash
    serves four consecutive elements: the noise of flat element i is bits
    16*(i mod 4) .. 16*(i mod 4)+15 of splitmix64(key + floor(i / 4))
    (mod 2**64).
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

_M64 = (1 << 64) - 1
_INC = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

MOMENT_FIRST = 0    # Muon momentum, AdamW exp_avg
MOMENT_SECOND = 1   # AdamW exp_avg_sq
MOMENT_PARAM = 2    # the parameter


def splitmix64(x):
    """SplitMix64 output from state x, for a Python int or a uint64 array."""
    if isinstance(x, (int, np.integer)):
        z = (int(x) + _INC) & _M64
        z = ((z ^ (z >> 30)) * _C1) & _M64
        z = ((z ^ (z >> 27)) * _C2) & _M64
        return z ^ (z >> 31)
    z = np.asarray(x, dtype=np.uint64) + np.uint64(_INC)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
    return z ^ (z >> np.uint64(31))


def sr_key(seed: int, stream: int) -> int:
    return splitmix64((int(seed) & _M64) ^ splitmix64(int(stream) & _M64))


def sr_stream(tensor_index: int, moment: int) -> int:
    return 4 * int(tensor_index) + int(moment)


def sr_noise16(key: int, index) -> np.ndarray:
    """16 uniform bits for each flat index (uint32 values in [0, 65536))."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        h = splitmix64(np.uint64(key) + (idx >> np.uint64(2)))
    shift = np.uint64(16) * (idx & np.uint64(3))
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
