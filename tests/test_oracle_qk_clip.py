"""Pins of the QK-Clip oracle (kimi-k3 "Optimization", "QK-Clip watches a
different failure mode"; dew.training.optim "scale_by_qk_clip").

The defining property: after the rescale, the maximum (scaled) query-key
score of a clipped head, measured again on the same inputs, equals the
threshold, and every other head's scores are unchanged. Scores are computed
here from the weights directly, not from the oracle's factors.
"""
import numpy as np
import pytest

import oracle
import synth

H, D, DM, T = 4, 16, 64, 12      # heads, head dim, model dim, positions


def _scores(x, Wq, Wk, h, d=D, q0=0, k0=0):
    """Causal max of (x Wq_h^T)(x Wk_h^T)^T / sqrt(d) for head h."""
    q = x @ Wq[q0 + h * d:q0 + (h + 1) * d].T
    k = x @ Wk[k0 + h * d:k0 + (h + 1) * d].T
    s = (q @ k.T) / np.sqrt(d)
    mask = np.tril(np.ones((len(x), len(x)), dtype=bool))
    return s[mask].max()


def _setup(seed):
    x = synth.normal(seed, 1, (T, DM)).astype(np.float64)
    Wq = synth.normal(seed, 2, (H * D, DM), std=0.5).astype(np.float64)
    Wk = synth.normal(seed, 3, (H * D, DM), std=0.5).astype(np.float64)
    Wq[:D] *= 3.0                    # head 0 runs hot
    return x, Wq, Wk


@pytest.mark.parametrize("alpha", [0.5, 0.3])
def test_clipped_heads_land_on_tau_and_others_stay(alpha):
    x, Wq, Wk = _setup(1)
    s = np.array([_scores(x, Wq, Wk, h) for h in range(H)])
    tau = float(np.median(s))        # about half the heads are above
    eq = oracle.ClipEntry(H, D, 0, D, 0, alpha)
    ek = oracle.ClipEntry(H, D, 0, D, 0, 1.0 - alpha)
    Wq2 = oracle.qk_clip(Wq, eq, s, tau)
    Wk2 = oracle.qk_clip(Wk, ek, s, tau)
    for h in range(H):
        s2 = _scores(x, Wq2, Wk2, h)
        if s[h] > tau:
            assert s2 == pytest.approx(tau, rel=1e-12), h
        else:
            assert s2 == s[h]
            np.testing.assert_array_equal(Wq2[h * D:(h + 1) * D], Wq[h * D:(h + 1) * D])


def test_mla_rotary_query_takes_the_whole_factor():
    """A head's score = nope part (q_C . k_C, both per head) + rotary part
    (q_R . k_R with k_R shared across heads). q_C, k_C take gamma^0.5, q_R
    takes gamma, the shared k_R nothing: the whole score scales by gamma."""
    rng_x = synth.normal(2, 1, (T, DM)).astype(np.float64)
    dn, dr = 12, 4
    # per head: query rows [nope, rope]; key rows [nope]; one shared rope key
    Wqb = synth.normal(2, 2, (H * (dn + dr), DM), std=0.5).astype(np.float64)
    Wkb = synth.normal(2, 3, (H * dn, DM), std=0.5).astype(np.float64)
    Wkr = synth.normal(2, 4, (dr, DM), std=0.5).astype(np.float64)

    def score(Wqb, Wkb, h):
        q = rng_x @ Wqb[h * (dn + dr):(h + 1) * (dn + dr)].T
        kn = rng_x @ Wkb[h * dn:(h + 1) * dn].T
        kr = rng_x @ Wkr.T
        s = (q[:, :dn] @ kn.T + q[:, dn:] @ kr.T) / np.sqrt(dn + dr)
        return s[np.tril(np.ones((T, T), dtype=bool))].max()

    s = np.array([score(Wqb, Wkb, h) for h in range(H)])
    tau = 0.5 * float(s.max())
    Wqb2 = oracle.qk_clip(Wqb, oracle.ClipEntry(H, dn + dr, 0, dn, 0, 0.5), s, tau)
    Wqb2 = oracle.qk_clip(Wqb2, oracle.ClipEntry(H, dn + dr, dn, dr, 0, 1.0), s, tau)
    Wkb2 = oracle.qk_clip(Wkb, oracle.ClipEntry(H, dn, 0, dn, 0, 0.5), s, tau)
    for h in range(H):
        want = min(s[h], tau)
        assert score(Wqb2, Wkb2, h) == pytest.approx(want, rel=1e-12)


def test_gamma_and_skip():
    g = oracle.gamma([50.0, 100.0, 200.0, 400.0], 100.0)
    np.testing.assert_array_equal(g, [1.0, 1.0, 0.5, 0.25])
    W = np.ones((8, 3))
    e = oracle.ClipEntry(2, 4, 1, 2, 0, 0.5)
    out = oracle.qk_clip(W, e, [400.0, 50.0], 100.0)
    np.testing.assert_array_equal(out[:, 0], [1, 0.5, 0.5, 1, 1, 1, 1, 1])
    np.testing.assert_array_equal(oracle.qk_clip(W, e, [400.0, 50.0], 100.0, skipped=True), W)
