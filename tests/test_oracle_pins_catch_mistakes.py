"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of an oracle function (a dropped
term, a flipped sign, a transposed operand, a swapped weight, a missing
factor), swaps the copy in for the real function with monkeypatch, and runs
the pins that guard that function. At least one of them must fail with an
assertion: a pin set that let the mistake through would not be pinning the
function. The mistakes exist only in this file, for the length of one test;
a control case first checks that every pin used here passes on the real
oracle.
"""
import importlib
import math

import numpy as np
import pytest

import oracle

# The submodules by name: the package re-exports functions that share some of
# their names (grad_control, qk_clip).
o_adamw = importlib.import_module("oracle.adamw")
o_bf16 = importlib.import_module("oracle.bf16")
o_gc = importlib.import_module("oracle.grad_control")
o_muon = importlib.import_module("oracle.muon")
o_nsb = importlib.import_module("oracle.ns_bf16")
o_qk = importlib.import_module("oracle.qk_clip")
o_sr = importlib.import_module("oracle.stochastic_round")
from tests import test_oracle_adamw as adam_pins
from tests import test_oracle_bf16 as bf16_pins
from tests import test_oracle_grad_control as gc_pins
from tests import test_oracle_ns as ns_pins
from tests import test_oracle_ns_bf16 as nsb_pins
from tests import test_oracle_qk_clip as qk_pins
from tests import test_oracle_sr as sr_pins
from tests import test_oracle_update as up_pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

_REAL_NS = o_muon.newton_schulz
_REAL_STEP_TENSOR = o_muon.muon_step_tensor
_REAL_STEP_VIEW = o_muon.muon_step_view


def _plant(monkeypatch, name, fn, *modules):
    """Replaces `name` in the oracle package and in each module that holds it."""
    monkeypatch.setattr(oracle, name, fn)
    for m in modules:
        monkeypatch.setattr(m, name, fn)


def _failing(pins):
    """Names of the pins that fail with an assertion."""
    failed = []
    for name, pin in pins:
        try:
            pin()
        except AssertionError:
            failed.append(name)
    return failed


# ---- the pins each function is guarded by ------------------------------------

NS_PINS = [
    ("spectral 8x8", lambda: ns_pins.test_spectral_pin((8, 8))),
    ("spectral 64x64", lambda: ns_pins.test_spectral_pin((64, 64))),
    ("spectral 33x97", lambda: ns_pins.test_spectral_pin((33, 97))),
    ("spectral 97x33", lambda: ns_pins.test_spectral_pin((97, 33))),
    ("spectral, 2 steps", lambda: ns_pins.test_spectral_pin_fewer_steps(2)),
    ("singular values", ns_pins.test_singular_values_follow_scalar_quintic),
    ("brute force 8x8", lambda: ns_pins.test_brute_force_tiny((8, 8))),
    ("brute force 6x4", lambda: ns_pins.test_brute_force_tiny((6, 4))),
    ("schedule, Polar Express scaling",
     lambda: ns_pins.test_schedule_spectral_pin((24, 40), 1.01, 0.0)),
]
# Operand-order mistakes only type-check on square matrices.
NS_SQUARE_PINS = [p for p in NS_PINS if p[0] in ("spectral 8x8", "spectral 64x64",
                                                  "brute force 8x8")]

MOMENTUM_PINS = [
    ("closed form, constant gradient", up_pins.test_momentum_closed_form_constant_grad),
    ("two Nesterov forms agree", up_pins.test_flaxchat_and_speedtronic_nesterov_forms_agree),
]

APPLY_PINS = [
    ("zero update is pure decay", up_pins.test_apply_zero_update_is_pure_decay),
    ("closed form 6x4", lambda: up_pins.test_apply_closed_form((6, 4))),
    ("closed form 4x6", lambda: up_pins.test_apply_closed_form((4, 6))),
    ("cautious decay mask and ties", up_pins.test_cautious_wd_mask_and_ties),
    ("cautious update mask and ties", up_pins.test_cautious_update_mask_and_ties),
]

NORMUON_PINS = [
    ("Frobenius norm kept", up_pins.test_normuon_preserves_frobenius_norm),
    ("first step equalises rows", up_pins.test_normuon_first_step_equalises_row_norms),
    ("state is a lerp", up_pins.test_normuon_state_is_lerp),
    ("floor above every moment", up_pins.test_normuon_floor_above_every_moment_is_the_identity),
    ("floor clamps small rows", up_pins.test_normuon_floor_clamps_only_the_small_rows),
]

ADAMW_PINS = [
    ("torch AdamW, wd 0.1", lambda: adam_pins.test_matches_torch_adamw_float64(0.1)),
    ("step-one closed form", adam_pins.test_step_one_closed_form),
    ("zero gradient is pure decay", adam_pins.test_zero_grad_zero_state_is_pure_decay),
]

GC_PINS = [
    ("torch clip_grad_norm_, 0.25", lambda: gc_pins.test_matches_torch_clip_grad_norm_fp64(0.25)),
    ("unscale by a power of two", gc_pins.test_unscale_by_a_power_of_two_is_exact),
    ("norm of ones", gc_pins.test_closed_form_norm_of_ones),
    ("inf skips the step", lambda: gc_pins.test_non_finite_gradient_skips_the_whole_step(np.inf)),
    ("nan skips the step", lambda: gc_pins.test_non_finite_gradient_skips_the_whole_step(np.nan)),
]

QK_PINS = [
    ("clipped heads land on tau", lambda: qk_pins.test_clipped_heads_land_on_tau_and_others_stay(0.5)),
    ("MLA rotary query", qk_pins.test_mla_rotary_query_takes_the_whole_factor),
    ("gamma and skip", qk_pins.test_gamma_and_skip),
]

SR_PINS = [
    ("fmix32 published values", sr_pins.test_fmix32_published_values),
    ("round-up probability", lambda: sr_pins.test_round_up_probability_is_the_dropped_fraction(
        0x3F808000)),
    ("representable values stay", sr_pins.test_representable_values_never_move),
]

VIEW_PINS = [
    ("views are independent", lambda: up_pins.test_views_are_independent_matrices({})),
    ("packed view differs from the whole", up_pins.test_packed_view_differs_from_whole_matrix),
    ("silent view left alone", up_pins.test_zero_gradient_view_is_left_alone_with_the_flag),
    ("silent view per view", up_pins.test_flag_is_per_view_in_a_packed_tensor),
]

BF16_PINS = [
    ("torch cast on float32 values", bf16_pins.test_matches_torch_on_float32_values),
    ("ties and near ties", bf16_pins.test_ties_and_near_ties_from_float64),
]


NS_STORED_PINS = [
    ("rounding off is the fp64 oracle", lambda: nsb_pins.test_rounding_off_is_the_fp64_oracle_bit_for_bit((33, 97))),
    ("rounding off, tall", lambda: nsb_pins.test_rounding_off_is_the_fp64_oracle_bit_for_bit((48, 16))),
    ("folded normalisation", lambda: nsb_pins.test_folded_normalisation_is_the_same_iteration((24, 40))),
    ("stored matrices are bf16", lambda: nsb_pins.test_stored_matrices_are_bf16_and_only_those(False)),
    ("stored matrices are bf16, folded", lambda: nsb_pins.test_stored_matrices_are_bf16_and_only_those(True)),
    ("copy stage", nsb_pins.test_copy_stage_moves_each_entry_by_half_a_spacing_at_most),
]
NS_STORED_SQUARE_PINS = [
    ("rounding off, square", lambda: nsb_pins.test_rounding_off_is_the_fp64_oracle_bit_for_bit((64, 64))),
    ("folded normalisation, square", lambda: nsb_pins.test_folded_normalisation_is_the_same_iteration((32, 32))),
]


def test_every_pin_passes_on_the_real_oracle():
    every = (NS_PINS + MOMENTUM_PINS + APPLY_PINS + NORMUON_PINS + ADAMW_PINS + GC_PINS + QK_PINS
             + SR_PINS + VIEW_PINS + BF16_PINS + NS_STORED_PINS + NS_STORED_SQUARE_PINS)
    assert _failing(every) == []


# ---- Newton-Schulz ---------------------------------------------------------------

def _ns_with(mistake):
    def ns(Q, steps=oracle.NS_STEPS, coeffs=oracle.NS_COEFFS, eps=oracle.NS_EPS, norm_scale=1.0):
        sched = o_muon.coeff_schedule(coeffs, steps)
        Q = np.asarray(Q, dtype=np.float64)
        tall = Q.shape[0] > Q.shape[1]
        T = Q.T if tall else Q
        norm = np.sqrt(np.sum(T * T))
        if mistake == "norm squared":
            norm = norm * norm
        if mistake == "norm_scale ignored":
            norm_scale = 1.0
        den = norm * norm_scale + eps
        X = T / den if den > 0 else np.zeros_like(T)
        for a, b, c in sched:
            if mistake == "sign of b":
                b = -b
            if mistake == "a and c swapped":
                a, c = c, a
            A = X.T @ X if mistake == "gram transposed" else X @ X.T
            P = b * A + (0.0 if mistake == "c term dropped" else c) * (A @ A)
            X = a * X + (X @ P if mistake == "product order" else P @ X)
        if mistake == "tall result reshaped, not transposed" and tall:
            return _REAL_NS(Q.T, steps, coeffs, eps, norm_scale).copy().reshape(Q.shape)
        return X.T.copy() if tall else X
    return ns


@pytest.mark.parametrize("mistake", ["norm squared", "norm_scale ignored", "sign of b",
                                     "a and c swapped", "c term dropped",
                                     "tall result reshaped, not transposed"])
def test_newton_schulz_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "newton_schulz", _ns_with(mistake), o_muon)
    assert _failing(NS_PINS), mistake


@pytest.mark.parametrize("mistake", ["gram transposed", "product order"])
def test_newton_schulz_operand_order_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "newton_schulz", _ns_with(mistake), o_muon)
    assert _failing(NS_SQUARE_PINS), mistake


# ---- Newton-Schulz with bf16 storage (the error model) ----------------------------

def _ns_stored_with(mistake):
    def ns(Q, steps=oracle.NS_STEPS, coeffs=oracle.NS_COEFFS, eps=oracle.NS_EPS, norm_scale=1.0,
           round_fn=oracle.round_bf16, fold_norm=False, trace=None):
        sched = o_muon.coeff_schedule(coeffs, steps)
        Q = np.asarray(Q, dtype=np.float64)
        tall = Q.shape[0] > Q.shape[1]
        T = Q.T if tall else Q
        den = np.sqrt(np.sum(T * T)) * norm_scale + eps
        s = 1.0 / den if den > 0 else 0.0
        X = round_fn(T) if fold_norm else round_fn(T / den if den > 0 else np.zeros_like(T))
        if trace:
            trace("X", 0, X)
        for k, (a, b, c) in enumerate(sched):
            first = fold_norm and k == 0
            sa = s if mistake == "fold scales A by s" else s * s
            G = X.T @ X if mistake == "gram transposed" else X @ X.T
            A = round_fn(sa * G if first else G)
            if trace:
                trace("A", k, A)
            P = b * A + c * (A @ A)
            if mistake != "P not rounded":
                P = round_fn(P)
            if trace:
                trace("P", k, P)
            X = s * (a * X + P @ X) if first else a * X + P @ X
            if k + 1 < len(sched) or mistake == "last X rounded":
                X = round_fn(X)
                if trace and k + 1 < len(sched):
                    trace("X", k + 1, X)
        return X.T.copy() if tall else X
    return ns


@pytest.mark.parametrize("mistake", ["fold scales A by s", "P not rounded", "last X rounded"])
def test_stored_newton_schulz_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "newton_schulz_stored", _ns_stored_with(mistake), o_nsb, nsb_pins)
    assert _failing(NS_STORED_PINS), mistake


def test_stored_newton_schulz_operand_order_mistake_is_caught(monkeypatch):
    _plant(monkeypatch, "newton_schulz_stored", _ns_stored_with("gram transposed"), o_nsb,
           nsb_pins)
    assert _failing(NS_STORED_SQUARE_PINS)


# ---- momentum and Nesterov ----------------------------------------------------------

def _momentum_with(mistake):
    def mom(B, G, mu, nesterov=True):
        B_new = mu * B + (1.0 if mistake == "(1 - mu) dropped" else 1.0 - mu) * G
        if not nesterov:
            return B_new, B_new.copy()
        if mistake == "lerp ends swapped":
            Q = B_new + mu * (G - B_new)
        elif mistake == "lerp from the old buffer":
            Q = G + mu * (B - G)
        else:
            Q = G + mu * (B_new - G)
        return B_new, Q
    return mom


@pytest.mark.parametrize("mistake", ["(1 - mu) dropped", "lerp ends swapped",
                                     "lerp from the old buffer"])
def test_momentum_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "momentum_nesterov", _momentum_with(mistake), o_muon)
    assert _failing(MOMENTUM_PINS), mistake


# ---- shape scale and the update -------------------------------------------------------

def test_inverted_shape_scale_is_caught(monkeypatch):
    _plant(monkeypatch, "shape_scale", lambda rows, cols, rule=0: max(1.0, cols / rows) ** 0.5,
           o_muon)
    pins = [(f"golden {c['rows']}x{c['cols']}", lambda c=c: up_pins.test_shape_scale(c))
            for c in up_pins.GOLD["shape_scale_cases"]]
    assert _failing(pins + APPLY_PINS)


def _apply_with(mistake):
    def apply(W, U, G, lr, wd, cautious=oracle.CAUTIOUS_OFF):
        r, c = W.shape
        s = max(1.0, (c / r) if mistake == "scale inverted" else (r / c)) ** 0.5
        if cautious == oracle.CAUTIOUS_OFF:
            decay = (1.0 - wd) if mistake == "decay without lr" else (1.0 - lr * wd)
            sign = 1.0 if mistake == "update sign" else -1.0
            return decay * W + sign * lr * s * U
        if cautious == oracle.CAUTIOUS_WD:
            g = s * U
            if mistake == "strict mask":
                mask = (g * W > 0).astype(np.float64)
            else:
                mask = (g * W >= 0).astype(np.float64)
            if mistake == "mask on the update":
                return W - lr * (g * mask + wd * W)
            return W - lr * (g + wd * W * mask)
        delta = lr * s * U if mistake == "decay left out of delta" else lr * wd * W + lr * s * U
        mask = (delta * G > 0).astype(np.float64)
        return W - mask * delta
    return apply


@pytest.mark.parametrize("mistake", ["scale inverted", "decay without lr", "update sign",
                                     "strict mask", "mask on the update",
                                     "decay left out of delta"])
def test_update_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "muon_apply", _apply_with(mistake), o_muon)
    assert _failing(APPLY_PINS), mistake


# ---- NorMuon and Muon+ -----------------------------------------------------------------

def _normuon_with(mistake):
    def nm(U, sm, beta2, eps=oracle.NORMUON_FLOOR):
        v = np.sum(U * U, axis=1) if mistake == "sum, not mean" else np.mean(U * U, axis=1)
        w = beta2 if mistake == "lerp weight swapped" else 1.0 - beta2
        sm_new = sm + w * (v - sm)
        f = np.maximum(sm_new, eps)
        row_scale = 1.0 / (f if mistake == "square root dropped" else np.sqrt(f))
        U1 = U * row_scale[:, None]
        if mistake == "norm not restored":
            return U1, sm_new
        kappa = np.sqrt(np.sum(U * U)) / max(np.sqrt(np.sum(U1 * U1)), oracle.NORMUON_FLOOR)
        return kappa * U1, sm_new
    return nm


@pytest.mark.parametrize("mistake", ["sum, not mean", "lerp weight swapped",
                                     "square root dropped", "norm not restored"])
def test_normuon_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "normuon", _normuon_with(mistake), o_muon)
    assert _failing(NORMUON_PINS), mistake


def _muon_plus_with(mistake):
    def mp(U, eps=oracle.NS_EPS):
        if mistake == "columns first":
            C = U / np.sqrt(np.sum(U * U, axis=0) + eps)[None, :]
            return C / np.sqrt(np.sum(C * C, axis=1) + eps)[:, None]
        R = U / (np.sqrt(np.sum(U * U, axis=1)) + eps)[:, None]
        return R / (np.sqrt(np.sum(R * R, axis=0)) + eps)[None, :]
    return mp


@pytest.mark.parametrize("mistake", ["columns first", "eps outside the square root"])
def test_muon_plus_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "muon_plus_row_col", _muon_plus_with(mistake), o_muon)
    assert _failing([("column norms closed form", up_pins.test_muon_plus_column_norms_closed_form)])


# ---- views and the inactive-expert rule ------------------------------------------------

def test_views_taken_as_one_matrix_is_caught(monkeypatch):
    def as_one(W, G, B, hp, views=1, lr_mult=1.0, wd=0.0, sm=None, skip_zero_grad=False):
        return _REAL_STEP_TENSOR(W, G, B, hp, 1, lr_mult, wd, None, skip_zero_grad)
    _plant(monkeypatch, "muon_step_tensor", as_one, o_muon)
    assert _failing(VIEW_PINS)


def test_silent_view_still_decayed_is_caught(monkeypatch):
    def no_skip(W, G, B, hp, lr_mult=1.0, wd=0.0, sm=None, skip_zero_grad=False):
        return _REAL_STEP_VIEW(W, G, B, hp, lr_mult, wd, sm, False)
    _plant(monkeypatch, "muon_step_view", no_skip, o_muon)
    assert _failing(VIEW_PINS)


# ---- AdamW ------------------------------------------------------------------------------

def _adamw_with(mistake):
    def step(W, G, m, v, lr, beta1, beta2, eps, wd, t):
        W, G, m, v = (np.asarray(x, dtype=np.float64) for x in (W, G, m, v))
        if mistake == "betas swapped":
            beta1, beta2 = beta2, beta1
        m_new = beta1 * m + (1.0 - beta1) * G
        v_new = beta2 * v + (1.0 - beta2) * G * G
        if mistake == "no bias correction":
            m_hat, v_hat = m_new, v_new
        else:
            m_hat, v_hat = m_new / (1.0 - beta1 ** t), v_new / (1.0 - beta2 ** t)
        den = np.sqrt(v_hat + eps) if mistake == "eps inside the root" else np.sqrt(v_hat) + eps
        if mistake == "decay after the update":
            return (W - lr * m_hat / den) * (1.0 - lr * wd), m_new, v_new
        return W * (1.0 - lr * wd) - lr * m_hat / den, m_new, v_new
    return step


@pytest.mark.parametrize("mistake", ["betas swapped", "no bias correction",
                                     "eps inside the root", "decay after the update"])
def test_adamw_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "adamw_step", _adamw_with(mistake), o_adamw)
    assert _failing(ADAMW_PINS), mistake


# ---- gradient control ---------------------------------------------------------------------

def _grad_control_with(mistake):
    def gc(grads, inv_loss_scale=1.0, max_norm=0.0):
        total, finite = 0.0, True
        for g in grads:
            u = np.asarray(g, dtype=np.float64).ravel()
            if mistake != "norm of the scaled gradients":
                u = u * inv_loss_scale
            if mistake != "non-finite ignored" and not np.all(np.isfinite(u)):
                finite = False
                continue
            total += float(np.dot(u, u))
        if not finite:
            return o_gc.GradControl(norm=math.nan, mult=0.0, skip=True)
        norm = total if mistake == "square root dropped" else math.sqrt(total)
        coef = 1.0
        if max_norm > 0.0:
            coef = min(1.0, max_norm / (norm + (0.0 if mistake == "no clip eps" else 1e-6)))
        return o_gc.GradControl(norm=norm, mult=inv_loss_scale * coef, skip=False)
    return gc


@pytest.mark.parametrize("mistake", ["norm of the scaled gradients", "non-finite ignored",
                                     "square root dropped", "no clip eps"])
def test_gradient_control_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "grad_control", _grad_control_with(mistake), o_gc)
    assert _failing(GC_PINS), mistake


# ---- QK-Clip ------------------------------------------------------------------------------

def test_qk_clip_mistakes_are_caught(monkeypatch):
    def gamma_inverted(s_max, tau):
        s = np.asarray(s_max, dtype=np.float64)
        return np.where(s > tau, s / tau, 1.0)
    _plant(monkeypatch, "gamma", gamma_inverted, o_qk)
    assert _failing(QK_PINS)


def test_qk_clip_exponent_ignored_is_caught(monkeypatch):
    real_gamma = o_qk.gamma

    def clip(W, entry, s_max, tau, skipped=False):
        W = np.array(W, dtype=np.float64, copy=True)
        if skipped:
            return W
        g = real_gamma(s_max, tau)
        for h in range(entry.heads):
            r0 = h * entry.head_stride + entry.row_offset
            W[r0:r0 + entry.scaled_rows] *= g[entry.head_index0 + h]
        return W
    _plant(monkeypatch, "qk_clip", clip, o_qk)
    assert _failing(QK_PINS)


# ---- stochastic rounding -------------------------------------------------------------------

def test_stochastic_rounding_mistakes_are_caught(monkeypatch):
    real = o_sr.round_bf16_with_noise

    def nearest(x, noise16):
        return real(x, np.full(np.shape(np.asarray(x)), 0x8000))
    _plant(monkeypatch, "round_bf16_with_noise", nearest, o_sr)
    assert _failing(SR_PINS)


def test_hash_constant_typo_is_caught(monkeypatch):
    def fmix(x):
        m = 0xFFFFFFFF
        if isinstance(x, (int, np.integer)):
            x = int(x) & m
            x ^= x >> 16
            x = (x * 0x85EBCA6B) & m
            x ^= x >> 13
            x = (x * 0xC2B2AE3D) & m     # one hex digit off
            return x ^ (x >> 16)
        return np.array([fmix(int(v)) for v in np.asarray(x).ravel()], dtype=np.uint64)
    _plant(monkeypatch, "fmix32", fmix, o_sr)
    assert _failing(SR_PINS)


# ---- bf16 storage rounding ----------------------------------------------------------------

def _bf16_with(mistake):
    def rnd(x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        if mistake == "double rounding through float32":
            x = x.astype(np.float32).astype(np.float64)
        bits = x.reshape(-1).view(np.uint64)
        drop = np.uint64(45)
        mask = (np.uint64(1) << drop) - np.uint64(1)
        low, kept = bits & mask, bits & ~mask
        half = np.uint64(1) << np.uint64(44)
        if mistake == "ties away from zero":
            up = low >= half
        else:
            lsb = (bits >> drop) & np.uint64(1)
            up = (low > half) | ((low == half) & (lsb == np.uint64(1)))
        out = (kept + np.where(up, np.uint64(1) << drop, np.uint64(0))).view(np.float64)
        return out.reshape(x.shape)
    return rnd


@pytest.mark.parametrize("mistake", ["ties away from zero", "double rounding through float32"])
def test_bf16_rounding_mistakes_are_caught(monkeypatch, mistake):
    _plant(monkeypatch, "round_bf16", _bf16_with(mistake), o_bf16)
    assert _failing(BF16_PINS), mistake


# ---- the order of the stages in one view's step ----------------------------------------------

def test_muon_plus_before_normuon_is_caught(monkeypatch):
    def step(W, G, B, hp, lr_mult=1.0, wd=0.0, sm=None, skip_zero_grad=False):
        W, G, B = (np.asarray(a, dtype=np.float64) for a in (W, G, B))
        B_new, Q = o_muon.momentum_nesterov(B, G, hp.momentum, hp.nesterov)
        U = o_muon.newton_schulz(Q, hp.ns_steps, hp.coeffs, hp.eps, hp.norm_scale)
        if hp.muon_plus:
            U = o_muon.muon_plus_row_col(U, hp.plus_eps)
        sm_new = None
        if hp.normuon:
            U, sm_new = o_muon.normuon(U, np.zeros(W.shape[0]) if sm is None else sm, hp.beta2,
                                       hp.normuon_eps)
        W_new = o_muon.muon_apply(W, U, G, hp.lr * lr_mult, wd, hp.cautious)
        return o_muon.ViewResult(W=W_new, B=B_new, U=U, sm=sm_new)
    _plant(monkeypatch, "muon_step_view", step, o_muon)
    assert _failing([("step composes its pieces", up_pins.test_full_view_step_composes_pieces)])


def test_moonlight_factor_on_the_short_side_is_caught(monkeypatch):
    real = o_muon.shape_scale

    def scale(rows, cols, rule=0):
        if rule == oracle.SHAPE_MOONLIGHT:
            return 0.2 * min(rows, cols) ** 0.5
        return real(rows, cols, rule)
    _plant(monkeypatch, "shape_scale", scale, o_muon)
    pins = [(f"Moonlight RMS {s}", lambda s=s: up_pins.test_moonlight_shape_factor_gives_update_rms_0_2(s))
            for s in [(64, 64), (48, 200), (200, 48)]]
    assert _failing(pins)
