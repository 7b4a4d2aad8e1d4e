"""Per-element parity bars of the GPU path against the fp64 oracle.

fp32 elementwise stages (Muon momentum, AdamW moments, fp32 AdamW
parameters) are checked element by element:

    |got - want| <= 1e-6 * |want| + atol

where atol is a first-order running bound on what the kernels' fp32
arithmetic may contribute, carried through the steps like the values
themselves. For one momentum step  B' = mu B + (1 - mu) G  in fp32:

    E' = mu E + d_mu (|B| + |G|) + 2u (mu |B| + (1 - mu) |G|) + g_rel (1 - mu) |G|

with u = 2^-24 (two roundings: the product and the fused add), d_mu the
absolute error of the fp32 constants mu and 1 - mu (1 - mu is exact in fp32
by Sterbenz's lemma, so both constants carry the same d_mu) and g_rel the
relative error of any factor the gradient is multiplied by on the device
(the global-norm clip). Where the two terms do not cancel, E stays below
4e-7 |B'|, so the bound is at most 1.4e-6 relative; where they cancel, E
keeps the bar at the size of the rounding of the terms, which is all that
fp32 arithmetic can promise. The AdamW bound follows the kernel's order of
operations the same way (see adamw_atol). A factor 2 covers the neglected
second-order terms.

bf16 parameters are stored by rounding, so the bar there is what the
Newton-Schulz bar (2e-2 relative Frobenius on U) allows after the rounding.
Let sigma_i = 2e-2 * lr * scale * rms(U) be the per-element size of that
error (spread evenly over the elements) and ulp_i the bf16 spacing at the
oracle's value:

* per element, |got - round(W64)| <= ulp_i + 10 sigma_i: at most one ulp
  from the oracle's own rounding, except near zero, where the bf16 grid is
  finer than the Newton-Schulz error itself;
* the fraction of elements that differ from round(W64) is at most 1.25x the
  flip rate the bar predicts, mean(min(1, E|delta_i| / ulp_i)) with
  E|delta_i| = sqrt(2/pi) sigma_i, plus 0.002;
* the update W_new - base (base = the decayed previous weight) is within
  1.25x of the relative Frobenius error those flips predict, plus 1e-3, of
  the oracle's rounded update; and the update's projection on the oracle's
  (a systematic scale error of the update) is within 1e-2 + 2e-2/sqrt(m),
  m = min(rows, cols): spread over m singular directions the Newton-Schulz
  error projects on the update only by about 1/sqrt(m) of its size, but on
  a view of rank one all of it is a scale error.
"""
from __future__ import annotations

import json
import os

import numpy as np

U32 = 2.0 ** -24
REL = 1e-6          # the fp32 stage bar
NS_BAR = 2e-2       # the Newton-Schulz output bar (relative Frobenius)
SAFETY = 2.0        # on the first-order fp32 bounds


def _scale_bar(shape, ns_bar: float = NS_BAR) -> float:
    m = min(shape) if len(shape) == 2 else 1
    return 1e-2 + ns_bar / np.sqrt(max(m, 1))


def _f32_err(x: float) -> float:
    return abs(float(np.float32(x)) - x)


def record(kind: str, what: str, **stats) -> None:
    """Appends one measured-error record to $MH_PARITY_LOG (if set)."""
    path = os.environ.get("MH_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"kind": kind, "what": what, **stats}) + "\n")


# ---- fp32 stages ----------------------------------------------------------------

def momentum_atol(B_prev, G, mu: float, E_prev=0.0, g_rel: float = 0.0):
    """Running bound after one momentum step from B_prev (oracle values)."""
    B_prev = np.abs(np.asarray(B_prev, dtype=np.float64))
    G = np.abs(np.asarray(G, dtype=np.float64))
    d_mu = _f32_err(mu)
    om = 1.0 - mu
    return (mu * E_prev + d_mu * (B_prev + G) + 2 * U32 * (mu * B_prev + om * G)
            + g_rel * om * G)


def adamw_atol(W, G, m, v, lr, b1, b2, eps, wd, t, E=(0.0, 0.0, 0.0), g_rel=0.0):
    """Running bounds (Em, Ev, Ew) after one AdamW step from the oracle's
    (W, m, v), in the kernel's order of operations:
        m' = b1 m + (1 - b1) g;  v' = b2 v + (1 - b2) g^2
        d = sqrt(v') * ibc2 + eps;  W' = W * (1 - lr wd) - (lr * ibc1) * (m' / d)
    with ibc1 = 1/(1 - b1^t) and ibc2 = 1/sqrt(1 - b2^t) each rounded to fp32
    once. Ew includes the final rounding of both sides (fp32 parameters)."""
    Em, Ev, Ew = E
    W = np.asarray(W, dtype=np.float64)
    g = np.abs(np.asarray(G, dtype=np.float64)) * (1.0 + g_rel)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    u = U32
    mn = b1 * m + (1 - b1) * np.asarray(G, dtype=np.float64)
    vn = b2 * v + (1 - b2) * g * g
    Em = (b1 * Em + _f32_err(b1) * (np.abs(m) + g) + 2 * u * (b1 * np.abs(m) + (1 - b1) * g)
          + g_rel * (1 - b1) * g)
    Ev = (b2 * Ev + _f32_err(b2) * (v + g * g) + 3 * u * (b2 * v + (1 - b2) * g * g)
          + 2 * g_rel * (1 - b2) * g * g)
    ibc1 = 1.0 / (1.0 - b1 ** t)
    ibc2 = 1.0 / np.sqrt(1.0 - b2 ** t)
    s = np.sqrt(vn)
    with np.errstate(divide="ignore", invalid="ignore"):
        Es = np.where(s > 0, np.minimum(Ev / (2 * s), np.sqrt(Ev)), np.sqrt(Ev)) + u * s
    d = s * ibc2 + eps
    Ed = ibc2 * Es + 3 * u * d
    r = mn / d
    Er = Em / d + np.abs(mn) * Ed / (d * d) + u * np.abs(r)
    lrb = lr * ibc1
    upd = lrb * r
    Eupd = lrb * Er + 3 * u * np.abs(upd)
    decay = 1.0 - lr * wd
    Wn = W * decay - upd
    Ew = (decay * Ew + (3 * u * lr * wd + u) * np.abs(W) + u * np.abs(W * decay) + Eupd
          + 2 * u * np.abs(Wn))
    return Em, Ev, Ew


def check_fp32(got, want, atol, what: str, rel: float = REL) -> dict:
    """Asserts |got - want| <= rel |want| + SAFETY * atol everywhere and
    returns the measured errors."""
    want = np.asarray(want, dtype=np.float64)
    atol = np.broadcast_to(np.asarray(atol, dtype=np.float64), want.shape).ravel()
    want = want.ravel()
    got = np.asarray(got, dtype=np.float64).ravel()
    err = np.abs(got - want)
    bound = rel * np.abs(want) + SAFETY * atol
    bad = ~(err <= bound)          # NaN counts as bad
    with np.errstate(divide="ignore", invalid="ignore"):
        relerr = np.where(want != 0, err / np.abs(want), np.where(err == 0, 0.0, np.inf))
        ratio = np.where(bound > 0, err / bound, np.where(err == 0, 0.0, np.inf))
    stats = {"n": int(want.size), "max_rel": float(np.max(relerr)) if want.size else 0.0,
             "p999_rel": float(np.quantile(relerr[np.isfinite(relerr)], 0.999))
             if want.size else 0.0,
             "frac_above_1e-6": float(np.mean(relerr > rel)) if want.size else 0.0,
             "max_err_over_bound": float(np.max(ratio)) if want.size else 0.0}
    record("fp32", what, **stats)
    if bad.any():
        k = int(np.argmax(ratio))
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {want.size} elements outside "
            f"{rel:g}|want| + {SAFETY:g} atol; worst at {k}: got {got[k]!r} want {want[k]!r} "
            f"atol {atol[k]:.3g} ({stats})")
    return stats


# ---- bf16 parameters -------------------------------------------------------------

def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits; subnormal spacing
    2^-133 near zero)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def check_bf16_param(got, W64, base, step_scale: float, U, what: str,
                     round_fn=None, ns_bar: float = NS_BAR) -> dict:
    """Checks a bf16 parameter after one step against the oracle.

    got: the GPU's bf16 parameter (as float64); W64: the oracle's value before
    rounding; base: the part of W64 that is not the update (the decayed
    previous weight); step_scale: lr * shape scale of the update; U: the
    oracle's Newton-Schulz output for this step (only its rms is used)."""
    import oracle
    round_fn = round_fn or oracle.round_bf16
    got = np.asarray(got, dtype=np.float64)
    W64 = np.asarray(W64, dtype=np.float64)
    Wr = round_fn(W64)
    ulp = bf16_ulp(Wr)
    ulp64 = bf16_ulp(W64)
    sig = ns_bar * step_scale * float(np.sqrt(np.mean(np.asarray(U, dtype=np.float64) ** 2)))
    diff = np.abs(got - Wr)
    bound = ulp + 10.0 * sig
    bad = ~(diff <= bound)
    flips = float(np.mean(got != Wr))
    e_abs = np.sqrt(2.0 / np.pi) * sig
    p = np.minimum(1.0, e_abs / ulp64)
    flip_pred = float(np.mean(p))
    # expected squared difference per element: flips of one ulp where the
    # grid is coarser than the error, the error itself where it is finer
    e2 = np.where(sig < ulp64, p * ulp64 ** 2, sig ** 2)
    dref = Wr - base
    nd = float(np.linalg.norm(dref))
    dw_pred = float(np.sqrt(np.sum(e2)) / nd) if nd > 0 else 0.0
    dw_err = float(np.linalg.norm((got - base) - dref) / nd) if nd > 0 else float(
        np.linalg.norm(got - base))
    proj = float(np.sum((got - Wr) * dref) / (nd * nd)) if nd > 0 else 0.0
    stats = {"n": int(W64.size), "max_ulps_from_rounded": float(np.max(diff / ulp)),
             "max_diff_over_bound": float(np.max(diff / bound)), "flip_frac": flips,
             "flip_pred_at_bar": flip_pred, "dw_rel": dw_err, "dw_pred_at_bar": dw_pred,
             "scale_bias": proj, "w_rel": float(np.linalg.norm(got - W64) / np.linalg.norm(W64))}
    record("bf16_param", what, **stats)
    if bad.any():
        k = int(np.argmax(diff / bound))
        raise AssertionError(f"{what}: {int(bad.sum())} elements more than one ulp + 10 sigma "
                             f"from round(W64); worst got {got.ravel()[k]!r} "
                             f"rounded oracle {Wr.ravel()[k]!r} ({stats})")
    assert flips <= 1.25 * flip_pred + 2e-3, (what, stats)
    assert dw_err <= 1.25 * dw_pred + 1e-3, (what, stats)
    assert abs(proj) <= _scale_bar(W64.shape, ns_bar), (what, stats)
    return stats


def check_f32_update(got, W64, base, what: str, ns_bar: float = NS_BAR) -> dict:
    """fp32 parameter after one step: the update got - base within the
    Newton-Schulz bar of the oracle's, relative Frobenius, and the
    parameter within 1e-3 of the oracle's unless the update itself is a
    large part of it (then the Newton-Schulz bar carried through)."""
    got = np.asarray(got, dtype=np.float64)
    W64 = np.asarray(W64, dtype=np.float64)
    dref = W64 - base
    nd = float(np.linalg.norm(dref))
    dw_err = float(np.linalg.norm((got - base) - dref) / nd) if nd > 0 else 0.0
    w_err = float(np.linalg.norm(got - W64) / np.linalg.norm(W64))
    w_bar = max(1e-3, ns_bar * nd / float(np.linalg.norm(W64)))
    proj = float(np.sum((got - W64) * dref) / (nd * nd)) if nd > 0 else 0.0
    stats = {"n": int(W64.size), "dw_rel": dw_err, "w_rel": w_err, "w_bar": w_bar,
             "scale_bias": proj}
    record("f32_param", what, **stats)
    assert dw_err < ns_bar, (what, stats)
    assert w_err < w_bar, (what, stats)
    assert abs(proj) <= _scale_bar(W64.shape, ns_bar), (what, stats)
    return stats
