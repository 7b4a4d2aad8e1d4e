"""fp64 CPU oracle of the Muon half of the hybrid step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this file; it
exists so that tests, the smoke check and the CPU baseline can compare the
CUDA library against a plain, slow, obviously correct statement of the method.

Every function is written from the method's own description, step by step,
in float64 NumPy. Matrix products use ``@`` (a library primitive) and nothing
is fused or reordered beyond what the description states.

Sources (page title, section):
  [SPD]  Speedtronic docs, "v2 optimizers": "Newton-Schulz", "Muon update",
         "Muon+", "Cautious updates".
  [FLX]  flaxchat, "Optimizer": "Muon Algorithm" steps 1-4.
  [KIMI] kimi-k3, "Optimization": "A tensor's storage shape can be misleading"
         (matrix views) and "Why treat a matrix differently?".

Readings taken where the pages are silent or ambiguous:
  * Frobenius normalisation is X = T / (||T||_F + eps) with eps = 1e-7 [SPD];
    flaxchat's Polar Express form X = g / (||g|| * 1.01) is norm_scale 1.01
    with eps 0, and its per-iteration coefficients a schedule of (a, b, c).
  * "tall" means rows > cols strictly; a square matrix is not transposed.
  * The shape scale uses the stored view's rows/cols: max(1, rows/cols)**0.5.
    [KIMI "Why treat a matrix differently?"] names the Moonlight shape factor
    as its trainer's default, but the formula did not survive on the page;
    the optional shape rule SHAPE_MOONLIGHT reads it as the published
    Moonlight rule 0.2 * sqrt(max(rows, cols)).
  * NorMuon [FLX step 3]: statistics per row of the stored view (mean over
    columns); state zero-initialised, no bias correction; the per-row factor
    is rsqrt(max(sm, normuon_eps)) (normuon_eps = 1e-10 unless the caller
    sets it) and "normalize" restores the Frobenius norm the update had before
    the per-row rescale (the norm ratio's denominator floored at 1e-10 only
    against division by zero).
  * Muon+ row_col [SPD]: rows to unit L2 norm, then columns, each with eps
    inside the square root; eps defaults to the NS eps (1e-7).
  * Order when several are on: NS -> NorMuon -> Muon+ -> apply.
  * Cautious mode 1 [FLX step 4]: the mask gates weight decay only and keeps
    entries where update * param >= 0. Cautious mode 2 [SPD]: the mask gates
    the whole observed update (decay included) and keeps entries where
    update * gradient > 0.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# [SPD "Newton-Schulz"]: quintic coefficients, five steps, eps.
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
NS_EPS = 1e-7
NORMUON_FLOOR = 1e-10

CAUTIOUS_OFF = 0
CAUTIOUS_WD = 1       # [FLX step 4]
CAUTIOUS_UPDATE = 2   # [SPD "Cautious updates"]

SHAPE_RATIO = 0       # [SPD "Muon update"]
SHAPE_MOONLIGHT = 1   # [KIMI "Why treat a matrix differently?"], reading above


@dataclass
class MuonHparams:
    lr: float = 0.02
    momentum: float = 0.95
    nesterov: bool = True
    eps: float = NS_EPS
    ns_steps: int = NS_STEPS
    coeffs: tuple = NS_COEFFS
    norm_scale: float = 1.0       # X = Q / (||Q|| * norm_scale + eps)
    normuon: bool = False
    beta2: float = 0.95
    muon_plus: bool = False
    plus_eps: float = NS_EPS
    cautious: int = CAUTIOUS_OFF
    normuon_eps: float = NORMUON_FLOOR
    shape_rule: int = SHAPE_RATIO


def momentum_nesterov(B: np.ndarray, G: np.ndarray, mu: float, nesterov: bool = True):
    """[SPD "Muon update"], [FLX step 1].

    B <- mu*B + (1-mu)*G, then the Nesterov form Q = lerp(G, B, mu) =
    G + mu*(B - G). Without Nesterov the update direction is B itself.
    Returns (B_new, Q).
    """
    B_new = mu * B + (1.0 - mu) * G
    if nesterov:
        Q = G + mu * (B_new - G)
    else:
        Q = B_new.copy()
    return B_new, Q


def coeff_schedule(coeffs, steps: int):
    """One (a, b, c) per step: a single triple repeated, or a sequence of
    `steps` triples taken in order."""
    c = np.asarray(coeffs, dtype=np.float64)
    if c.shape == (3,):
        return [tuple(c)] * steps
    if c.shape != (steps, 3):
        raise ValueError(f"need one (a, b, c) or {steps} of them, got shape {c.shape}")
    return [tuple(r) for r in c]


def newton_schulz(Q: np.ndarray, steps: int = NS_STEPS, coeffs=NS_COEFFS,
                  eps: float = NS_EPS, norm_scale: float = 1.0) -> np.ndarray:
    """[SPD "Newton-Schulz"]: quintic iteration on one matrix.

    A tall matrix (rows > cols) is transposed, normalised, iterated and
    transposed back. Each step forms A = X X^T and X <- a X + (b A + c A^2) X.

    The normalisation is X = T / (||T||_F * norm_scale + eps): Speedtronic's
    form with norm_scale 1 and eps 1e-7; flaxchat's Polar Express (step 2,
    X <- g / (||g|| * 1.01), then one (a, b, c) per iteration from a list)
    with norm_scale 1.01, eps 0 and a coefficient schedule. A zero matrix
    stays zero (with eps 0 the division is skipped).
    """
    sched = coeff_schedule(coeffs, steps)
    Q = np.asarray(Q, dtype=np.float64)
    tall = Q.shape[0] > Q.shape[1]
    T = Q.T if tall else Q
    den = np.sqrt(np.sum(T * T)) * norm_scale + eps
    X = T / den if den > 0 else np.zeros_like(T)
    for a, b, c in sched:
        A = X @ X.T
        P = b * A + c * (A @ A)
        X = a * X + P @ X
    return X.T.copy() if tall else X


def normuon(U: np.ndarray, sm: np.ndarray, beta2: float, eps: float = NORMUON_FLOOR):
    """[FLX step 3] NorMuon per-row second moment (reading: rows of the stored view).

    v_i = mean_j U_ij^2; sm <- lerp(sm, v, 1 - beta2); each row is scaled by
    rsqrt(max(sm_i, eps)); then the whole matrix is rescaled so that its
    Frobenius norm equals the norm U had before the per-row scaling (the
    ratio's denominator floored at 1e-10). Returns (U_new, sm_new).
    """
    v = np.mean(U * U, axis=1)
    sm_new = sm + (1.0 - beta2) * (v - sm)
    row_scale = 1.0 / np.sqrt(np.maximum(sm_new, eps))
    U1 = U * row_scale[:, None]
    norm_before = np.sqrt(np.sum(U * U))
    norm_after = np.sqrt(np.sum(U1 * U1))
    kappa = norm_before / max(norm_after, NORMUON_FLOOR)
    return kappa * U1, sm_new


def muon_plus_row_col(U: np.ndarray, eps: float = NS_EPS) -> np.ndarray:
    """[SPD "Muon+"] row_col mode: normalise rows, then columns, eps inside each sqrt."""
    R = U / np.sqrt(np.sum(U * U, axis=1) + eps)[:, None]
    return R / np.sqrt(np.sum(R * R, axis=0) + eps)[None, :]


def shape_scale(rows: int, cols: int, rule: int = SHAPE_RATIO) -> float:
    """[SPD "Muon update"]: max(1, rows/cols)^0.5 of the stored view; with
    SHAPE_MOONLIGHT, 0.2 * max(rows, cols)^0.5."""
    if rule == SHAPE_MOONLIGHT:
        return 0.2 * max(rows, cols) ** 0.5
    if rule != SHAPE_RATIO:
        raise ValueError(f"unknown shape rule {rule}")
    return max(1.0, rows / cols) ** 0.5


def muon_apply(W: np.ndarray, U: np.ndarray, G: np.ndarray, lr: float, wd: float,
               cautious: int = CAUTIOUS_OFF, shape_rule: int = SHAPE_RATIO) -> np.ndarray:
    """Parameter update of one view, fp64.

    Plain [SPD]: W <- (1 - lr*wd) W - lr * s * U, s = shape_scale(rows, cols, shape_rule).
    Cautious mode 1 [FLX step 4], with g = s*U the update direction:
        mask = (g * W >= 0);  W <- W - lr * (g + wd * W * mask).
    Cautious mode 2 [SPD "Cautious updates"], the observed update of the plain
    rule being delta = lr*wd*W + lr*s*U:
        mask = (delta * G > 0);  W <- W - mask * delta.
    """
    s = shape_scale(W.shape[0], W.shape[1], shape_rule)
    if cautious == CAUTIOUS_OFF:
        return (1.0 - lr * wd) * W - lr * s * U
    if cautious == CAUTIOUS_WD:
        g = s * U
        mask = (g * W >= 0).astype(np.float64)
        return W - lr * (g + wd * W * mask)
    if cautious == CAUTIOUS_UPDATE:
        delta = lr * wd * W + lr * s * U
        mask = (delta * G > 0).astype(np.float64)
        return W - mask * delta
    raise ValueError(f"unknown cautious mode {cautious}")


@dataclass
class ViewResult:
    W: np.ndarray
    B: np.ndarray
    U: np.ndarray
    sm: np.ndarray | None = None


def muon_step_view(W, G, B, hp: MuonHparams, lr_mult: float = 1.0, wd: float = 0.0,
                   sm=None, skip_zero_grad: bool = False) -> ViewResult:
    """One Muon update of one r x c view, in the pages' order:
    momentum + Nesterov -> Newton-Schulz -> [NorMuon] -> [Muon+] -> apply.

    skip_zero_grad [KIMI "One more kind of state: which experts learn?";
    "A tensor's storage shape can be misleading": unselected experts with no
    gradient are not quietly decayed]: a view whose gradient is zero
    everywhere is left as it is -- parameter, momentum and NorMuon state --
    and its update direction is zero.
    """
    W = np.asarray(W, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if skip_zero_grad and not np.any(G):
        keep_sm = None
        if hp.normuon:
            keep_sm = np.zeros(W.shape[0]) if sm is None else np.asarray(sm, np.float64).copy()
        return ViewResult(W=W.copy(), B=B.copy(), U=np.zeros_like(W), sm=keep_sm)
    B_new, Q = momentum_nesterov(B, G, hp.momentum, hp.nesterov)
    U = newton_schulz(Q, hp.ns_steps, hp.coeffs, hp.eps, hp.norm_scale)
    sm_new = None
    if hp.normuon:
        U, sm_new = normuon(U, np.zeros(W.shape[0]) if sm is None else np.asarray(sm, np.float64),
                            hp.beta2, hp.normuon_eps)
    if hp.muon_plus:
        U = muon_plus_row_col(U, hp.plus_eps)
    lr = hp.lr * lr_mult
    W_new = muon_apply(W, U, G, lr, wd, hp.cautious, hp.shape_rule)
    return ViewResult(W=W_new, B=B_new, U=U, sm=sm_new)


def muon_step_tensor(W, G, B, hp: MuonHparams, views: int = 1, lr_mult: float = 1.0,
                     wd: float = 0.0, sm=None, skip_zero_grad: bool = False):
    """[KIMI "storage shape"]: a packed tensor declared as (views, r, c) is
    ``views`` independent r x c matrices sharing one momentum buffer.

    W, G, B are arrays of total size views*r*c (any shape); they are viewed
    as (views, r, c). Returns (W_new, B_new, U, sm_new) shaped like the input
    (U and sm as (views, r, c) and (views, r)).
    """
    W = np.asarray(W, dtype=np.float64)
    shape = W.shape
    r, c = shape[-2], shape[-1]
    if views > 1 and W.ndim == 2:
        r = shape[0] // views
    Wv = W.reshape(views, r, c)
    Gv = np.asarray(G, dtype=np.float64).reshape(views, r, c)
    Bv = np.asarray(B, dtype=np.float64).reshape(views, r, c)
    smv = None if sm is None else np.asarray(sm, dtype=np.float64).reshape(views, r)
    Wn = np.empty_like(Wv)
    Bn = np.empty_like(Bv)
    Un = np.empty_like(Wv)
    smn = np.empty((views, r)) if hp.normuon else None
    for k in range(views):
        res = muon_step_view(Wv[k], Gv[k], Bv[k], hp, lr_mult, wd,
                             None if smv is None else smv[k], skip_zero_grad)
        Wn[k], Bn[k], Un[k] = res.W, res.B, res.U
        if hp.normuon:
            smn[k] = res.sm
    return Wn.reshape(shape), Bn.reshape(shape), Un, smn
