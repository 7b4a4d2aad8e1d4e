"""Pins for the oracle's momentum, apply, NorMuon, Muon+, cautious and view logic (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "muon_update.json")))


def _n(seed, tid, shape):
    return synth.normal(seed, tid, shape).astype(np.float64)


# --- momentum + Nesterov (Speedtronic "Muon update"; flaxchat step 1) ---------

def test_momentum_closed_form_constant_grad():
    # Constant G from a zero buffer: B_k = (1 - mu^k) G and the Nesterov
    # lerp gives Q_k = (1 - mu^(k+1)) G.
    G = _n(0, 1, (5, 7))
    mu = 0.95
    Bk = np.zeros_like(G)
    for k in range(1, 8):
        Bk, Q = oracle.momentum_nesterov(Bk, G, mu, True)
        np.testing.assert_allclose(Bk, (1 - mu ** k) * G, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(Q, (1 - mu ** (k + 1)) * G, rtol=1e-13, atol=1e-15)


def test_momentum_without_nesterov_uses_buffer():
    G, B0 = _n(0, 2, (3, 4)), _n(0, 3, (3, 4))
    B1, Q = oracle.momentum_nesterov(B0, G, 0.9, False)
    np.testing.assert_array_equal(Q, B1)


def test_flaxchat_and_speedtronic_nesterov_forms_agree():
    # flaxchat writes g <- g(1-b) + m b; Speedtronic writes lerp(g, B, b).
    G, B0 = _n(1, 2, (6, 3)), _n(1, 3, (6, 3))
    mu = 0.95
    B1, Q = oracle.momentum_nesterov(B0, G, mu, True)
    np.testing.assert_allclose(Q, G * (1 - mu) + B1 * mu, rtol=1e-14, atol=1e-16)


# --- apply / shape scale (Speedtronic "Muon update") ----------------------------

@pytest.mark.parametrize("case", GOLD["shape_scale_cases"])
def test_shape_scale(case):
    assert oracle.shape_scale(case["rows"], case["cols"]) == pytest.approx(case["scale"], rel=1e-15)


@pytest.mark.parametrize("shape", [(64, 64), (48, 200), (200, 48), (1, 9), (9, 1)])
def test_moonlight_shape_factor_gives_update_rms_0_2(shape):
    """kimi-k3 "Why treat a matrix differently?": the Moonlight shape factor,
    read as Moonlight's published rule, scales an update whose singular
    values are all one (full rank) to an RMS of 0.2 for any shape. U is built
    by QR here, independently of the Newton-Schulz oracle."""
    r, c = shape
    rng = np.random.default_rng(r * 1000 + c)
    Qm, _ = np.linalg.qr(rng.standard_normal((max(r, c), min(r, c))))
    U = Qm if r >= c else Qm.T
    W = np.zeros(shape)
    lr = 0.5
    out = oracle.muon_apply(W, U, U, lr, 0.0, shape_rule=oracle.SHAPE_MOONLIGHT)
    rms = np.sqrt(np.mean((out / lr) ** 2))
    assert rms == pytest.approx(0.2, rel=1e-12)
    # the ratio rule instead gives RMS max(1, r/c)^0.5 / sqrt(max(r, c))
    out = oracle.muon_apply(W, U, U, lr, 0.0)
    assert np.sqrt(np.mean((out / lr) ** 2)) == pytest.approx(
        max(1.0, r / c) ** 0.5 / max(r, c) ** 0.5, rel=1e-12)


def test_apply_zero_update_is_pure_decay():
    W = _n(2, 1, (6, 4))
    out = oracle.muon_apply(W, np.zeros_like(W), np.zeros_like(W), lr=0.02, wd=0.01)
    np.testing.assert_array_equal(out, (1 - 0.02 * 0.01) * W)


@pytest.mark.parametrize("shape", [(6, 4), (4, 6), (5, 5)])
def test_apply_closed_form(shape):
    W, U = _n(2, 2, shape), _n(2, 3, shape)
    lr, wd = 0.02, 0.01
    out = oracle.muon_apply(W, U, U, lr, wd)
    s = max(1.0, shape[0] / shape[1]) ** 0.5
    np.testing.assert_allclose(out - (1 - lr * wd) * W, -lr * s * U, rtol=1e-12, atol=1e-15)


def test_cautious_wd_mask_and_ties():
    # flaxchat step 4: mask = (g * param >= 0), param -= lr (g + wd param mask).
    W = np.array([[1.0, -1.0, 2.0, 0.0, 3.0]])
    U = np.array([[0.5, 0.5, -0.5, 0.7, 0.0]])  # ties: W = 0 and U = 0 -> mask 1
    lr, wd = 0.1, 0.5
    out = oracle.muon_apply(W, U, np.ones_like(W), lr, wd, oracle.CAUTIOUS_WD)
    mask = np.array([[1, 0, 0, 1, 1]], dtype=np.float64)
    s = 1.0
    want = W - lr * (s * U + wd * W * mask)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


def test_cautious_update_mask_and_ties():
    # Speedtronic "Cautious updates": mask = (observed_update * gradient > 0),
    # parameter = old - masked_update; the update includes weight decay.
    W = np.array([[1.0, -1.0, 2.0, 0.0, 3.0, 1.0]])
    U = np.array([[0.5, 0.5, -0.5, 0.0, 0.0, -0.05]])
    G = np.array([[1.0, 1.0, 1.0, 1.0, 0.0, 1.0]])  # G = 0 tie -> masked out
    lr, wd = 0.1, 0.5
    out = oracle.muon_apply(W, U, G, lr, wd, oracle.CAUTIOUS_UPDATE)
    delta = lr * wd * W + lr * U
    keep = (delta * G > 0)
    want = np.where(keep, W - delta, W)
    np.testing.assert_array_equal(out, want)
    assert out[0, 3] == 0.0 and out[0, 4] == 3.0  # zero delta / zero grad: unchanged


# --- NorMuon (flaxchat step 3, reading: per row of the stored view) ------------

def test_normuon_preserves_frobenius_norm():
    U = _n(3, 1, (12, 20))
    sm = np.abs(_n(3, 2, (12,))) * 0.01
    out, sm_new = oracle.normuon(U, sm, 0.95)
    assert np.linalg.norm(out) == pytest.approx(np.linalg.norm(U), rel=1e-13)


def test_normuon_first_step_equalises_row_norms():
    U = _n(3, 3, (9, 31)) * np.linspace(0.1, 3.0, 9)[:, None]
    out, sm_new = oracle.normuon(U, np.zeros(9), 0.95)
    row_norms = np.linalg.norm(out, axis=1)
    np.testing.assert_allclose(row_norms, row_norms[0], rtol=1e-12)
    np.testing.assert_allclose(sm_new, 0.05 * np.mean(U * U, axis=1), rtol=1e-14)


def test_normuon_state_is_lerp():
    U = _n(3, 4, (4, 6))
    sm = np.abs(_n(3, 5, (4,)))
    _, sm_new = oracle.normuon(U, sm, 0.9)
    v = np.mean(U * U, axis=1)
    np.testing.assert_allclose(sm_new, 0.9 * sm + 0.1 * v, rtol=1e-14)


def test_normuon_floor_above_every_moment_is_the_identity():
    # With the floor above every row's second moment all rows get the same
    # factor 1/sqrt(eps), and restoring the Frobenius norm undoes it exactly.
    U = _n(3, 6, (7, 11)) * np.linspace(0.2, 4.0, 7)[:, None]
    out, sm_new = oracle.normuon(U, np.zeros(7), 0.95, eps=1e6)
    np.testing.assert_allclose(out, U, rtol=1e-13)
    np.testing.assert_allclose(sm_new, 0.05 * np.mean(U * U, axis=1), rtol=1e-14)


def test_normuon_floor_clamps_only_the_small_rows():
    # Rows whose moment is under the floor keep their relative size; rows above
    # it are equalised. Row 0 is tiny (moment 1e-8), rows 1.. are O(1).
    U = _n(3, 7, (5, 40))
    U[0] *= 1e-4
    eps = 1e-4
    out, sm_new = oracle.normuon(U, np.zeros(5), 0.0, eps=eps)
    f = 1.0 / np.sqrt(np.maximum(sm_new, eps))
    assert f[0] == pytest.approx(1.0 / np.sqrt(eps))
    U1 = U * f[:, None]
    kappa = np.linalg.norm(U) / np.linalg.norm(U1)
    np.testing.assert_allclose(out, kappa * U1, rtol=1e-13)
    big = np.linalg.norm(out[1:], axis=1)
    np.testing.assert_allclose(big, big[0], rtol=1e-12)


def test_normuon_zero_update_stays_zero():
    out, sm_new = oracle.normuon(np.zeros((3, 5)), np.zeros(3), 0.95)
    assert np.all(out == 0) and np.all(np.isfinite(out)) and np.all(sm_new == 0)


# --- Muon+ (Speedtronic "Muon+") ------------------------------------------------

def test_muon_plus_column_norms_closed_form():
    U = _n(4, 1, (10, 14))
    eps = 1e-3
    out = oracle.muon_plus_row_col(U, eps)
    R = U / np.sqrt(np.sum(U * U, axis=1, keepdims=True) + eps)
    s = np.sum(R * R, axis=0)
    np.testing.assert_allclose(np.linalg.norm(out, axis=0), np.sqrt(s / (s + eps)), rtol=1e-13)
    # rows are normalised first: before the column step every row norm is
    # sqrt(r2 / (r2 + eps))
    r2 = np.sum(U * U, axis=1)
    np.testing.assert_allclose(np.linalg.norm(R, axis=1), np.sqrt(r2 / (r2 + eps)), rtol=1e-13)


def test_muon_plus_zero_stays_zero():
    out = oracle.muon_plus_row_col(np.zeros((4, 4)), 1e-7)
    assert np.all(out == 0)


# --- matrix views (kimi-k3 "A tensor's storage shape can be misleading") -------

@pytest.mark.parametrize("flags", [dict(), dict(normuon=True), dict(muon_plus=True, cautious=1),
                                   dict(cautious=2)])
def test_views_are_independent_matrices(flags):
    hp = oracle.MuonHparams(**flags)
    k, r, c = 2, 12, 5
    W, G = _n(5, 1, (k * r, c)), _n(5, 2, (k * r, c))
    B = _n(5, 3, (k * r, c)) * 0.1
    Wn, Bn, U, sm = oracle.muon_step_tensor(W, G, B, hp, views=k, wd=0.01)
    for v in range(k):
        rs = slice(v * r, (v + 1) * r)
        one = oracle.muon_step_view(W[rs], G[rs], B[rs], hp, wd=0.01)
        np.testing.assert_array_equal(Wn[rs], one.W)
        np.testing.assert_array_equal(Bn[rs], one.B)


def test_packed_view_differs_from_whole_matrix():
    hp = oracle.MuonHparams()
    W, G = _n(6, 1, (16, 6)), _n(6, 2, (16, 6))
    B = np.zeros_like(W)
    as_views, _, _, _ = oracle.muon_step_tensor(W, G, B, hp, views=2)
    whole, _, _, _ = oracle.muon_step_tensor(W, G, B, hp, views=1)
    assert np.abs(as_views - whole).max() > 1e-4


def test_full_view_step_composes_pieces():
    hp = oracle.MuonHparams(normuon=True, muon_plus=True, cautious=1)
    W, G, B = _n(7, 1, (9, 13)), _n(7, 2, (9, 13)), _n(7, 3, (9, 13))
    res = oracle.muon_step_view(W, G, B, hp, lr_mult=0.5, wd=0.1)
    B1, Q = oracle.momentum_nesterov(B, G, hp.momentum)
    U = oracle.newton_schulz(Q)
    U, _ = oracle.normuon(U, np.zeros(9), hp.beta2)
    U = oracle.muon_plus_row_col(U, hp.plus_eps)
    np.testing.assert_array_equal(res.W, oracle.muon_apply(W, U, G, hp.lr * 0.5, 0.1, 1))


# ---- inactive experts (kimi-k3 "Optimization", "One more kind of state: which
# experts learn?": an expert that received no gradient acquires no momentum and
# no weight decay) ------------------------------------------------------------

def _expert(seed):
    W = synth.normal(seed, 1, (24, 40)).astype(np.float64)
    B = synth.normal(seed, 2, (24, 40), std=1e-2).astype(np.float64)
    return W, B


def test_zero_gradient_view_is_left_alone_with_the_flag():
    W, B = _expert(50)
    for hp in (oracle.MuonHparams(), oracle.MuonHparams(normuon=True)):
        sm = np.full(24, 0.3)
        r = oracle.muon_step_view(W, np.zeros_like(W), B, hp, 1.0, 0.1, sm, skip_zero_grad=True)
        np.testing.assert_array_equal(r.W, W)
        np.testing.assert_array_equal(r.B, B)
        assert np.all(r.U == 0)
        if hp.normuon:
            np.testing.assert_array_equal(r.sm, sm)


def test_without_the_flag_a_zero_gradient_view_still_moves():
    """The closed form the flag prevents: B <- mu B, and the step runs on
    Q = mu B with decay (1 - lr wd)."""
    W, B = _expert(51)
    hp = oracle.MuonHparams()
    r = oracle.muon_step_view(W, np.zeros_like(W), B, hp, 1.0, 0.1)
    np.testing.assert_allclose(r.B, hp.momentum * B, rtol=1e-15)
    U = oracle.newton_schulz(hp.momentum * hp.momentum * B)
    want = (1 - hp.lr * 0.1) * W - hp.lr * U     # 24 x 40: shape scale 1
    np.testing.assert_allclose(r.W, want, rtol=1e-12, atol=1e-15)


def test_flag_does_not_touch_views_with_any_gradient():
    W, B = _expert(52)
    G = np.zeros_like(W)
    G[3, 7] = 1e-3                                 # one routed token is enough
    hp = oracle.MuonHparams()
    a = oracle.muon_step_view(W, G, B, hp, 1.0, 0.1, skip_zero_grad=True)
    b = oracle.muon_step_view(W, G, B, hp, 1.0, 0.1)
    np.testing.assert_array_equal(a.W, b.W)
    np.testing.assert_array_equal(a.B, b.B)


def test_flag_is_per_view_in_a_packed_tensor():
    """A packed (2, r, c) tensor with one silent view: only that view stays."""
    W = synth.normal(53, 1, (2 * 24, 40)).astype(np.float64)
    B = synth.normal(53, 2, (2 * 24, 40), std=1e-2).astype(np.float64)
    G = synth.normal(53, 3, (2 * 24, 40), std=1e-3).astype(np.float64)
    G[:24] = 0.0
    hp = oracle.MuonHparams()
    Wn, Bn, _, _ = oracle.muon_step_tensor(W, G, B, hp, views=2, wd=0.1, skip_zero_grad=True)
    np.testing.assert_array_equal(Wn[:24], W[:24])
    np.testing.assert_array_equal(Bn[:24], B[:24])
    ref = oracle.muon_step_view(W[24:], G[24:], B[24:], hp, 1.0, 0.1)
    np.testing.assert_array_equal(Wn[24:], ref.W)
