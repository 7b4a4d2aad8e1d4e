"""Pins for the bf16-storage model of the Newton-Schulz iteration (CPU only).

oracle.ns_bf16.newton_schulz_stored is the quintic iteration with X, A and P
stored through a rounding function. Its pins:

* with rounding off it is the fp64 oracle bit for bit (which is itself pinned
  to the SVD of its input), and with the normalisation folded into the first
  step's products it still equals U p^5(Sigma) V^T from numpy's SVD;
* every matrix it stores is bf16-representable, and nothing else is rounded
  (the returned X of the last step is not);
* its error follows the unit roundoff: rounding to p significant bits gives an
  error that shrinks by about 2^4 for every 4 more bits;
* one stage that only copies X (a = 1, b = c = 0) changes each entry by at most
  half a bf16 spacing, 2^-8 relative (8 significant bits);
* on N(0, 1) inputs it lands about 1 % from the fp64 iteration, inside the
  2e-2 Newton-Schulz bar.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle.ns_bf16 import newton_schulz_stored, round_to_bits
from synth import spectra
from tests.test_oracle_ns import spectral_expected

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _ident(x):
    return x


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("shape", [(16, 48), (48, 16), (64, 64), (33, 97), (1, 7)])
def test_rounding_off_is_the_fp64_oracle_bit_for_bit(shape):
    Q = synth.normal(11, shape[0] * 131 + shape[1], shape).astype(np.float64)
    got = newton_schulz_stored(Q, round_fn=_ident)
    assert np.array_equal(got, oracle.newton_schulz(Q))
    sched = [(3.4445, -4.775, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    got = newton_schulz_stored(Q, steps=3, coeffs=sched, eps=0.0, norm_scale=1.01,
                               round_fn=_ident)
    assert np.array_equal(got, oracle.newton_schulz(Q, 3, sched, 0.0, 1.01))


@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (32, 32)])
def test_folded_normalisation_is_the_same_iteration(shape):
    Q = 3.7 * synth.normal(12, shape[0] + shape[1], shape).astype(np.float64)
    got = newton_schulz_stored(Q, round_fn=_ident, fold_norm=True)
    assert _rel(got, spectral_expected(Q)) < 1e-11


def test_zero_matrix_stays_zero():
    Z = np.zeros((8, 24))
    for fold in (False, True):
        assert np.array_equal(newton_schulz_stored(Z, fold_norm=fold), Z)
        assert np.array_equal(newton_schulz_stored(Z, eps=0.0, fold_norm=fold), Z)


@pytest.mark.parametrize("fold", [False, True])
def test_stored_matrices_are_bf16_and_only_those(fold):
    Q = synth.normal(13, 5, (48, 80)).astype(np.float64)
    seen = []

    def trace(name, k, M):
        seen.append((name, k))
        assert np.array_equal(oracle.round_bf16(M), M), (name, k)
    out = newton_schulz_stored(Q, fold_norm=fold, trace=trace)
    assert seen == [("X", 0)] + [(n, k + 1 if n == "X" else k)
                                 for k in range(5) for n in "APX"][:-1]
    # The last X is returned as computed, not stored: it is not on the bf16 grid.
    assert not np.array_equal(oracle.round_bf16(out), out)


def test_round_to_bits_8_is_bf16_rounding():
    x = synth.normal(14, 1, (4096,)).astype(np.float64) * 10.0 ** np.linspace(-20, 20, 4096)
    assert np.array_equal(round_to_bits(8)(x), oracle.round_bf16(x))


def test_error_follows_the_unit_roundoff():
    Q = spectra.matrix("gaussian", 64, 160, seed=3).astype(np.float64)
    ref = oracle.newton_schulz(Q)
    errs = {p: _rel(newton_schulz_stored(Q, round_fn=round_to_bits(p)), ref) for p in (8, 12, 16)}
    for lo, hi in ((8, 12), (12, 16)):
        ratio = errs[lo] / errs[hi]
        assert 2.0 ** 3 < ratio < 2.0 ** 5, (errs, ratio)
    assert 2.0 ** -9 < errs[8] < 2.0 ** -5, errs


def test_copy_stage_moves_each_entry_by_half_a_spacing_at_most():
    Q = synth.normal(15, 2, (40, 72)).astype(np.float64)
    X0 = Q / (np.linalg.norm(Q) + 1e-7)
    got = newton_schulz_stored(Q, steps=1, coeffs=(1.0, 0.0, 0.0))
    # X1 = 1 * round(X0) + round(0 * A + 0 * A A) X = round(X0)
    assert np.all(np.abs(got - X0) <= 2.0 ** -8 * np.abs(X0))
    assert np.array_equal(got, oracle.round_bf16(X0))


@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (128, 128)])
def test_gaussian_inputs_land_inside_the_ns_bar(shape):
    Q = spectra.matrix("gaussian", *shape, seed=4).astype(np.float64)
    err = _rel(newton_schulz_stored(Q, fold_norm=True), oracle.newton_schulz(Q))
    assert 2e-3 < err < 2e-2, err
