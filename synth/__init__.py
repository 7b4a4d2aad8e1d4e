"""Seeded synthetic inputs, shared by the CPU oracle side and the CUDA side.

This module holds no optimizer arithmetic. It only turns (seed, tensor_id,
flat index) into numbers, so that the fp64 oracle and the GPU kernels can be
fed bit-identical inputs without either one producing the other's data.

Generator (defined here, implemented twice: NumPy below, CUDA in synth.cu):

* ``splitmix64(x)``: Steele/Lea/Flood's SplitMix64 finaliser on the 64-bit
  counter ``x`` (wrapping arithmetic).
* per-tensor key: ``key = splitmix64(seed ^ splitmix64(tensor_id))``.
* element ``i`` draws six words ``w_k = splitmix64(key + 6*i + k)``,
  ``k = 0..5``, and sums their twelve 32-bit halves into ``S`` (exact in
  64-bit integers, ``S < 12 * 2**32``).
* ``z = float32((S - 6 * 2**32) * 2**-32)``: the Irwin-Hall(12) approximation
  of a standard normal (mean 0, variance 1, support [-6, 6]). The subtraction
  and the power-of-two scale are exact in float64; the one rounding is the
  float64 -> float32 round-to-nearest-even.
* ``x = z * std`` in float32 (one IEEE multiply), optionally rounded to bf16
  by round-to-nearest-even.

Every step is integer arithmetic or a single correctly rounded IEEE
operation, so both implementations give the same bits on any host or GPU.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "splitmix64_int",
    "tensor_key",
    "normal_f32",
    "normal",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "lognormal_factor",
    "CHUNK",
]

_MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
CHUNK = 1 << 22


def splitmix64_int(x: int) -> int:
    """SplitMix64 on one Python integer (mod 2**64)."""
    z = (x + _GOLDEN) & _MASK64
    z = ((z ^ (z >> 30)) * _MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * _MIX2) & _MASK64
    return z ^ (z >> 31)


def _splitmix64_vec(x: np.ndarray) -> np.ndarray:
    z = x + np.uint64(_GOLDEN)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
    return z ^ (z >> np.uint64(31))


def tensor_key(seed: int, tensor_id: int) -> int:
    return splitmix64_int((seed & _MASK64) ^ splitmix64_int(tensor_id & _MASK64))


def normal_f32(seed: int, tensor_id: int, count: int, offset: int = 0,
               std: float | np.float32 = 1.0) -> np.ndarray:
    """``count`` float32 draws for flat indices ``offset .. offset+count-1``."""
    key = np.uint64(tensor_key(seed, tensor_id))
    std32 = np.float32(std)
    out = np.empty(count, dtype=np.float32)
    lo_mask = np.uint64(0xFFFFFFFF)
    shift = np.uint64(32)
    bias = np.int64(6 << 32)
    for start in range(0, count, CHUNK):
        n = min(CHUNK, count - start)
        idx = np.arange(offset + start, offset + start + n, dtype=np.uint64)
        base = key + idx * np.uint64(6)
        s = np.zeros(n, dtype=np.uint64)
        for k in range(6):
            w = _splitmix64_vec(base + np.uint64(k))
            s += (w & lo_mask) + (w >> shift)
        z = ((s.astype(np.int64) - bias).astype(np.float64) * (2.0 ** -32)).astype(np.float32)
        out[start:start + n] = z * std32
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = ((b & np.uint64(0x7F800000)) == np.uint64(0x7F800000)) & ((b & np.uint64(0x7FFFFF)) != 0)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(nan, (b >> np.uint64(16)) | np.uint64(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(seed: int, tensor_id: int, shape, std: float | np.float32 = 1.0,
           dtype: str = "f32", offset: int = 0) -> np.ndarray:
    """Draws shaped as ``shape`` (row-major). ``dtype='bf16'`` returns the
    bf16-rounded values widened to float32 (exactly representable)."""
    count = int(np.prod(shape)) if len(shape) else 1
    x = normal_f32(seed, tensor_id, count, offset=offset, std=std)
    if dtype == "bf16":
        x = bf16_bits_to_f32(f32_to_bf16_bits(x))
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return x.reshape(shape)


def lognormal_factor(seed: int, tensor_id: int) -> np.float32:
    """One per-tensor factor exp(z), z the tensor's draw at a reserved id.

    Computed once on the host in float64 and rounded to float32; both sides
    receive this same float32 as part of their ``std``.
    """
    z = float(normal_f32(seed, (tensor_id ^ 0x5A5A5A5A) + (1 << 40), 1)[0])
    return np.float32(math.exp(z))
