"""The parity bars themselves, on the CPU (tests.parity, tests.helpers).

A simulated GPU step stands in for the device: the Newton-Schulz output from
the bf16-storage model of the iteration (oracle.ns_bf16, folded as the
kernels fold the normalisation), the momentum replayed in float32 in the
kernel's order of operations, the parameter update computed from that U and
rounded to the parameter's dtype. The bars must pass on it, and fail on a
planted mistake: an update scaled by 3 %, one wrong parameter element, a
momentum off by 1e-5 relative on a hundred elements, a moment without its
(1 - beta) factor.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.helpers import check_muon_views, oracle_muon_tensor
from tests.parity import adamw_atol, check_bf16_param, check_fp32

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

F = np.float32


def _wl(param_dtype, rows=384, cols=1024, views=2, **hp):
    spec = W.MuonSpec("t", views, rows, cols, param_dtype, "bf16")
    return W.Workload("sim", muon=[spec], adamw=[], muon_hp=dict(W.MUON_HP, **hp),
                      adam_hp=dict(W.ADAM_HP), steps=1)


def _simulated_step(wl, scale=1.0):
    """(W, B) of one simulated device step of the workload's tensor 0."""
    spec = wl.muon[0]
    hp = wl.muon_hp
    r, c = spec.rows, spec.cols
    Ws, Bs = [], []
    for v in range(spec.views):
        off = v * r * c
        W0 = W.host_tensor(wl, W.KIND_W, 0, offset=off, count=r * c).reshape(r, c)
        G = W.host_tensor(wl, W.KIND_G, 0, offset=off, count=r * c).reshape(r, c)
        mu = F(hp["momentum"])
        B = (mu * np.zeros((r, c), F) + (F(1) - mu) * G.astype(F)).astype(np.float64)
        Q = (G.astype(F) + mu * (B.astype(F) - G.astype(F))).astype(np.float64)
        U = oracle.newton_schulz_stored(Q, fold_norm=True)
        lr = hp["lr"] * spec.lr_mult
        s = oracle.shape_scale(r, c)
        Wn = (1 - lr * spec.wd) * W0 - scale * lr * s * U
        Ws.append(oracle.round_bf16(Wn) if spec.param_dtype == "bf16"
                  else Wn.astype(F).astype(np.float64))
        Bs.append(B)
    return np.stack(Ws), np.stack(Bs)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bars_pass_on_a_simulated_device_step(dtype):
    wl = _wl(dtype)
    got_w, got_b = _simulated_step(wl)
    ref = oracle_muon_tensor(wl, 0, 1)
    check_muon_views(wl, 0, ref, got_w, got_b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_a_three_percent_update_scale_error_fails(dtype):
    wl = _wl(dtype)
    got_w, got_b = _simulated_step(wl, scale=1.03)
    ref = oracle_muon_tensor(wl, 0, 1)
    with pytest.raises(AssertionError):
        check_muon_views(wl, 0, ref, got_w, got_b)


def test_one_wrong_bf16_parameter_element_fails():
    wl = _wl("bf16")
    got_w, got_b = _simulated_step(wl)
    ref = oracle_muon_tensor(wl, 0, 1)
    got_w[1, 17, 300] += 3 * oracle.round_bf16(np.array([abs(got_w[1, 17, 300])]))[0] * 2 ** -7
    with pytest.raises(AssertionError):
        check_muon_views(wl, 0, ref, got_w, got_b)


def test_momentum_off_on_a_hundred_elements_fails():
    wl = _wl("bf16")
    got_w, got_b = _simulated_step(wl)
    ref = oracle_muon_tensor(wl, 0, 1)
    idx = np.random.default_rng(0).choice(got_b[0].size, 100, replace=False)
    got_b[0].reshape(-1)[idx] *= 1 + 1e-5
    with pytest.raises(AssertionError):
        check_muon_views(wl, 0, ref, got_w, got_b)


def test_adamw_moment_without_its_factor_fails():
    n = 1 << 16
    g = np.random.default_rng(1).standard_normal(n) * 1e-3
    w = np.random.default_rng(2).standard_normal(n) * 0.02
    z = np.zeros(n)
    _, m, _ = oracle.adamw_step(w, g, z, z, 3e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    em, _, _ = adamw_atol(w, g, z, z, 3e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    m32 = (F(0.9) * z.astype(F) + (F(1) - F(0.9)) * g.astype(F)).astype(np.float64)
    check_fp32(m32, m, em, "simulated m")
    with pytest.raises(AssertionError):
        check_fp32(g.astype(F).astype(np.float64), m, em, "m without (1 - beta1)")


def test_bf16_bar_allows_the_zero_crossing_and_counts_flips():
    """Near zero the bf16 grid is finer than the Newton-Schulz error: a value
    many spacings from the rounded oracle there is accepted, the same
    distance on a large value is not."""
    W64 = np.array([1e-6, 0.5, -0.25, 0.125] * 64)
    base = W64 + 1e-4
    U = np.ones_like(W64)
    got = oracle.round_bf16(W64)
    got[0] = oracle.round_bf16(np.array([W64[0] + 2e-6]))[0]
    check_bf16_param(got, W64, base, 1e-4, U, "zero crossing")
    got[1] = oracle.round_bf16(np.array([W64[1] + 2e-2]))[0]
    with pytest.raises(AssertionError):
        check_bf16_param(got, W64, base, 1e-4, U, "large value off")
