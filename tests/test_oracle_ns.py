"""Pins for the oracle's Newton-Schulz iteration (CPU only).

Each test ties oracle.newton_schulz to something other than itself:
the SVD of its input (numpy.linalg.svd), invariances any correct
implementation must have, and a brute-force loop on tiny inputs.
The coefficients come from the page's printed values in tests/golden.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ns_coefficients.json")))
A, B, C = GOLD["a"], GOLD["b"], GOLD["c"]
STEPS, EPS = GOLD["steps"], GOLD["eps"]

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def quintic_k(sigma, k):
    """The scalar quintic p(s) = a s + b s^3 + c s^5 applied k times."""
    s = np.asarray(sigma, dtype=np.float64)
    for _ in range(k):
        s = A * s + B * s ** 3 + C * s ** 5
    return s


def spectral_expected(Q, steps=STEPS, eps=EPS):
    """U p^k(Sigma) V^T from the SVD of Q / (||Q||_F + eps)."""
    Q = np.asarray(Q, dtype=np.float64)
    X = Q / (np.linalg.norm(Q) + eps)
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    return (U * quintic_k(s, steps)[None, :]) @ Vt


def test_defaults_match_printed_coefficients():
    assert oracle.NS_COEFFS == (A, B, C)
    assert oracle.NS_STEPS == STEPS
    assert oracle.NS_EPS == EPS


@pytest.mark.parametrize("shape", [(8, 8), (16, 48), (48, 16), (64, 64), (33, 97), (97, 33),
                                   (128, 512), (512, 128), (1, 7), (7, 1)])
def test_spectral_pin(shape):
    Q = synth.normal(1, 100 + shape[0] * 1000 + shape[1], shape).astype(np.float64)
    got = oracle.newton_schulz(Q)
    want = spectral_expected(Q)
    err = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert err < 1e-11, err


@pytest.mark.parametrize("steps", [1, 2, 3])
def test_spectral_pin_fewer_steps(steps):
    Q = synth.normal(2, 7, (24, 40)).astype(np.float64)
    got = oracle.newton_schulz(Q, steps=steps)
    want = spectral_expected(Q, steps=steps)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-12


def test_singular_values_follow_scalar_quintic():
    Q = synth.normal(3, 1, (40, 90)).astype(np.float64)
    s_in = np.linalg.svd(Q / (np.linalg.norm(Q) + EPS), compute_uv=False)
    s_out = np.linalg.svd(oracle.newton_schulz(Q), compute_uv=False)
    np.testing.assert_allclose(np.sort(s_out), np.sort(np.abs(quintic_k(s_in, STEPS))),
                               rtol=1e-10, atol=1e-13)


def test_singular_vectors_match_svd_polar_factor():
    # A well-spread spectrum: every sigma/||Q|| is large enough that five
    # quintic steps keep it positive, so the output shares U V^T's singular
    # vectors and NS(Q) (U V^T)^T is symmetric positive definite.
    rng = np.random.default_rng(0)
    U, _ = np.linalg.qr(rng.standard_normal((20, 20)))
    V, _ = np.linalg.qr(rng.standard_normal((50, 20)))
    s = np.linspace(1.0, 2.0, 20)
    Q = (U * s) @ V.T
    out = oracle.newton_schulz(Q)
    polar = U @ V.T
    M = out @ polar.T
    np.testing.assert_allclose(M, M.T, atol=1e-12)
    assert np.all(np.linalg.eigvalsh((M + M.T) / 2) > 0.5)
    # Not exactly orthogonal: the iteration is approximate (kimi-k3
    # "Optimization": singular values are not all exactly one).
    sv = np.linalg.svd(out, compute_uv=False)
    assert sv.min() > 0.6 and sv.max() < 1.25
    assert np.abs(sv - 1).max() > 1e-3


def test_zero_matrix_stays_zero_and_finite():
    for shape in [(4, 9), (9, 4), (5, 5)]:
        out = oracle.newton_schulz(np.zeros(shape))
        assert np.all(np.isfinite(out))
        assert np.all(out == 0)


def test_tall_is_transpose_of_wide():
    Q = synth.normal(4, 2, (70, 30)).astype(np.float64)
    np.testing.assert_array_equal(oracle.newton_schulz(Q), oracle.newton_schulz(Q.T).T)


def test_square_transpose_equivariance():
    Q = synth.normal(4, 3, (30, 30)).astype(np.float64)
    np.testing.assert_allclose(oracle.newton_schulz(Q.T), oracle.newton_schulz(Q).T,
                               atol=1e-12)


def test_scale_invariance():
    # NS(alpha Q) with eps scaled by alpha equals NS(Q): only the ratio
    # ||Q|| / eps enters the normalisation.
    Q = synth.normal(5, 1, (20, 36)).astype(np.float64)
    base = oracle.newton_schulz(Q)
    for alpha in (1e-3, 0.5, 7.0, 1e4):
        np.testing.assert_allclose(oracle.newton_schulz(alpha * Q, eps=alpha * EPS), base,
                                   atol=1e-12)
    # With eps fixed the dependence on scale is only through eps.
    np.testing.assert_allclose(oracle.newton_schulz(1e4 * Q), base, atol=1e-7)


def test_orthogonal_equivariance():
    rng = np.random.default_rng(1)
    Q = synth.normal(6, 1, (12, 30)).astype(np.float64)
    P, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    R, _ = np.linalg.qr(rng.standard_normal((30, 30)))
    np.testing.assert_allclose(oracle.newton_schulz(P @ Q @ R), P @ oracle.newton_schulz(Q) @ R,
                               atol=1e-12)


def test_rank_preserved():
    rng = np.random.default_rng(2)
    Q = rng.standard_normal((40, 3)) @ rng.standard_normal((3, 64))
    sv = np.linalg.svd(oracle.newton_schulz(Q), compute_uv=False)
    assert np.all(sv[:3] > 0.3)
    assert np.all(sv[3:] < 1e-9)


def _brute_ns(Q, steps, eps):
    """Triple-loop restatement on Python floats (tiny inputs only)."""
    r, c = len(Q), len(Q[0])
    tall = r > c
    T = [[Q[j][i] for j in range(r)] for i in range(c)] if tall else [row[:] for row in Q]
    m, n = len(T), len(T[0])
    norm = sum(T[i][j] ** 2 for i in range(m) for j in range(n)) ** 0.5
    X = [[T[i][j] / (norm + eps) for j in range(n)] for i in range(m)]
    for _ in range(steps):
        Am = [[sum(X[i][k] * X[j][k] for k in range(n)) for j in range(m)] for i in range(m)]
        A2 = [[sum(Am[i][k] * Am[k][j] for k in range(m)) for j in range(m)] for i in range(m)]
        P = [[B * Am[i][j] + C * A2[i][j] for j in range(m)] for i in range(m)]
        X = [[A * X[i][j] + sum(P[i][k] * X[k][j] for k in range(m)) for j in range(n)]
             for i in range(m)]
    if tall:
        return [[X[j][i] for j in range(m)] for i in range(n)]
    return X


@pytest.mark.parametrize("shape", [(3, 5), (8, 8), (6, 4), (1, 1), (2, 8)])
def test_brute_force_tiny(shape):
    Q = synth.normal(7, shape[0] * 10 + shape[1], shape).astype(np.float64)
    want = np.array(_brute_ns(Q.tolist(), STEPS, EPS))
    np.testing.assert_allclose(oracle.newton_schulz(Q), want, rtol=1e-12, atol=1e-14)


# ---- coefficient schedules and the Polar Express normalisation ---------------------
# flaxchat "Optimizer", "Muon Algorithm" step 2: X <- g / (||g|| * 1.01), then one
# (a, b, c) per iteration from a list. The page prints no coefficient values, so
# the schedules below are arbitrary; the pins hold for any schedule.

SCHED = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.6, -2.4, 0.8), (2.0, -1.5, 0.5),
         (1.875, -1.25, 0.375)]


def spectral_schedule(Q, sched, eps, norm_scale):
    """U (p_k o ... o p_1)(Sigma) V^T from the SVD of Q / (||Q|| * norm_scale + eps),
    p_i(s) = a_i s + b_i s^3 + c_i s^5 applied in the schedule's order."""
    Q = np.asarray(Q, dtype=np.float64)
    U, s, Vt = np.linalg.svd(Q / (np.linalg.norm(Q) * norm_scale + eps), full_matrices=False)
    for a, b, c in sched:
        s = a * s + b * s ** 3 + c * s ** 5
    return (U * s[None, :]) @ Vt


@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (32, 32), (5, 17)])
@pytest.mark.parametrize("norm_scale,eps", [(1.0, EPS), (1.01, 0.0)])
def test_schedule_spectral_pin(shape, norm_scale, eps):
    Q = synth.normal(9, shape[0] * 100 + shape[1], shape).astype(np.float64)
    got = oracle.newton_schulz(Q, steps=len(SCHED), coeffs=SCHED, eps=eps, norm_scale=norm_scale)
    want = spectral_schedule(Q, SCHED, eps, norm_scale)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-11


def test_schedule_order_matters_and_constant_schedule_is_the_triple():
    Q = synth.normal(9, 1, (20, 36)).astype(np.float64)
    fwd = oracle.newton_schulz(Q, steps=5, coeffs=SCHED)
    rev = oracle.newton_schulz(Q, steps=5, coeffs=SCHED[::-1])
    assert np.linalg.norm(fwd - rev) / np.linalg.norm(fwd) > 1e-3
    const = oracle.newton_schulz(Q, steps=5, coeffs=[(A, B, C)] * 5)
    np.testing.assert_array_equal(const, oracle.newton_schulz(Q))


def test_polar_express_normalisation_keeps_zero_and_scales():
    Z = np.zeros((6, 9))
    out = oracle.newton_schulz(Z, steps=5, coeffs=SCHED, eps=0.0, norm_scale=1.01)
    assert np.all(out == 0)
    Q = synth.normal(9, 2, (12, 30)).astype(np.float64)
    # with eps 0 the normalised input is scale-free: NS(alpha Q) == NS(Q)
    a = oracle.newton_schulz(Q, steps=5, coeffs=SCHED, eps=0.0, norm_scale=1.01)
    b = oracle.newton_schulz(1e3 * Q, steps=5, coeffs=SCHED, eps=0.0, norm_scale=1.01)
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-12
    # and its largest input singular value is 1/1.01 of the Frobenius-normalised one
    s = np.linalg.svd(Q / (np.linalg.norm(Q) * 1.01), compute_uv=False)
    assert s[0] < 1.0 / 1.01 + 1e-15


def test_schedule_length_must_match_steps():
    with pytest.raises(ValueError):
        oracle.newton_schulz(np.eye(4), steps=3, coeffs=SCHED)
