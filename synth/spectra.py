"""Seeded matrices with a prescribed singular spectrum.

Inputs only; no optimizer arithmetic. A matrix ``U diag(s) V^T`` is built
from orthonormal factors taken from the QR factorisation of seeded normal
draws (``synth.normal``) and a spectrum ``s`` given in closed form, then
rounded to float32 so that the GPU and the oracle read the same values.

Spectra (``kind``), for an r x c matrix with m = min(r, c):
* ``rank_deficient``: the first m/4 values evenly spaced in [0.5, 1], the
  rest exactly zero (before the float32 rounding);
* ``low_rank_noise``: eight values equal to 1, the rest 1e-3 (a rank-8
  signal plus a flat noise floor);
* ``decaying``: s_k = 10^(-4 k / (m - 1)), four decades from the largest to
  the smallest;
* ``gaussian``: no construction, the plain N(0, 1) draws the other tests use.
"""
from __future__ import annotations

import numpy as np

from . import normal

KINDS = ("rank_deficient", "low_rank_noise", "decaying")


def spectrum(kind: str, m: int) -> np.ndarray:
    k = np.arange(m, dtype=np.float64)
    if kind == "rank_deficient":
        r = max(1, m // 4)
        s = np.zeros(m)
        s[:r] = np.linspace(1.0, 0.5, r)
        return s
    if kind == "low_rank_noise":
        s = np.full(m, 1e-3)
        s[:min(8, m)] = 1.0
        return s
    if kind == "decaying":
        return 10.0 ** (-4.0 * k / max(m - 1, 1))
    raise ValueError(kind)


def _orthonormal(seed: int, tensor_id: int, n: int, m: int) -> np.ndarray:
    g = normal(seed, tensor_id, (n, m)).astype(np.float64)
    q, r = np.linalg.qr(g)
    return q * np.sign(np.diag(r))[None, :]


def matrix(kind: str, rows: int, cols: int, seed: int = 0, tensor_id: int = 0) -> np.ndarray:
    """float32 (rows, cols) matrix with singular values spectrum(kind, m)."""
    if kind == "gaussian":
        return normal(seed, tensor_id, (rows, cols))
    m = min(rows, cols)
    U = _orthonormal(seed, 2 * tensor_id + 1000003, rows, m)
    V = _orthonormal(seed, 2 * tensor_id + 1000004, cols, m)
    return ((U * spectrum(kind, m)[None, :]) @ V.T).astype(np.float32)
