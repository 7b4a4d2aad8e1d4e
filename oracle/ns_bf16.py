"""Newton-Schulz with bf16 storage of its iterates: an error model.

TEST INFRASTRUCTURE ONLY; the product path never imports it.

The pages run the quintic iteration (Speedtronic docs, "v2 optimizers",
"Newton-Schulz"; flaxchat, "Optimizer", "Muon Algorithm" step 2) in plain
PyTorch without fixing the precision of the iterates. The fp64 oracle
(oracle.muon.newton_schulz) is the reference. A tensor-core implementation
keeps X, A = X X^T and P = b A + c A^2 in bf16 between its products and
accumulates each product in fp32. This function is the same iteration, step
for step and in the same operation order as the fp64 oracle, with those three
stored matrices passed through ``round_fn`` right after they are formed:

    X = round(T / (||T||_F * norm_scale + eps))
    repeat:  A = round(X X^T);  P = round(b A + c (A A));  X = a X + P X
             (X rounded again except after the last step)

The products themselves are exact (fp64): fp32 accumulation adds about
2^-24 sqrt(K) relative, far below bf16's unit roundoff 2^-8. The last X is
returned unrounded, as the fused update consumes it in fp32. With
``round_fn = lambda x: x`` the result equals the fp64 oracle bit for bit.

What it is for: the difference between this and the fp64 oracle is the
error that bf16 storage alone causes, so it predicts the size of the GPU
path's error on any input (well-spread, low-rank or strongly decaying
spectra). It does not predict the GPU's values: a GPU run and this model
round different values (the GPU rounds Q before it scales by 1/||Q||, and
sums in a different order), and on decaying spectra the iteration amplifies
each rounding pattern differently.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16
from .muon import NS_COEFFS, NS_EPS, NS_STEPS, coeff_schedule


def newton_schulz_stored(Q: np.ndarray, steps: int = NS_STEPS, coeffs=NS_COEFFS,
                         eps: float = NS_EPS, norm_scale: float = 1.0, round_fn=round_bf16,
                         fold_norm: bool = False, trace=None) -> np.ndarray:
    """The quintic iteration with X, A and P stored through ``round_fn``.

    ``fold_norm``: store T itself (unscaled) as the first X and apply the
    normalisation s = 1 / (||T||_F * norm_scale + eps) inside the first
    step's products instead, A = round(s^2 X X^T) and X = round(s (a X + P X)),
    which is where a kernel that never re-reads T to scale it applies s.
    Mathematically the same iteration; it changes which values are rounded.

    ``trace(name, step, matrix)``, if given, sees every stored matrix
    ("X", "A", "P") as it is stored."""
    sched = coeff_schedule(coeffs, steps)
    Q = np.asarray(Q, dtype=np.float64)
    tall = Q.shape[0] > Q.shape[1]
    T = Q.T if tall else Q
    den = np.sqrt(np.sum(T * T)) * norm_scale + eps
    s = 1.0 / den if den > 0 else 0.0
    if fold_norm:
        X = round_fn(T)
    else:
        X = T / den if den > 0 else np.zeros_like(T)
        X = round_fn(X)
    if trace:
        trace("X", 0, X)
    for k, (a, b, c) in enumerate(sched):
        first = fold_norm and k == 0
        A = round_fn((s * s) * (X @ X.T) if first else X @ X.T)
        if trace:
            trace("A", k, A)
        P = round_fn(b * A + c * (A @ A))
        if trace:
            trace("P", k, P)
        X = s * (a * X + P @ X) if first else a * X + P @ X
        if k + 1 < len(sched):
            X = round_fn(X)
            if trace:
                trace("X", k + 1, X)
    return X.T.copy() if tall else X


def round_to_bits(bits: int):
    """Round to nearest (ties to even) keeping ``bits`` significand bits:
    bits = 8 is bf16 without its exponent limits. For checking that the
    model's error follows the unit roundoff 2^-bits."""
    def fn(x):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)                  # x = m 2^e, 0.5 <= |m| < 1
        return np.ldexp(np.round(np.ldexp(m, bits)), e - bits)
    return fn
