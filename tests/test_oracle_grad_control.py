"""Pins of the gradient-control oracle (global norm, clip factor, overflow skip).

kimi-k3 "Optimization", "Keep the arithmetic and gradients under control":
one global gradient norm, a clip when max_grad_norm > 0, the norm observed
when it is 0, and the whole hybrid update skipped on an FP16 overflow;
dew.training.optim "build_optimizer": the clip reads every gradient of every
parameter group together.
"""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _grads(seed, shapes, scale=1.0):
    rng = np.random.default_rng(seed)
    return [scale * rng.standard_normal(s) for s in shapes]


SHAPES = [(7, 5), (3, 11), (64,), (2, 4, 6)]


@pytest.mark.parametrize("max_norm_frac", [0.25, 0.999, 1.5, 10.0])
def test_matches_torch_clip_grad_norm_fp64(max_norm_frac):
    """PyTorch's clip_grad_norm_ (a library routine) in float64 on CPU:
    same total norm, same clipped gradients."""
    torch = pytest.importorskip("torch")
    gs = _grads(1, SHAPES, 0.3)
    norm = math.sqrt(sum(float((g * g).sum()) for g in gs))
    max_norm = max_norm_frac * norm
    params = []
    for g in gs:
        p = torch.zeros(g.shape, dtype=torch.float64, requires_grad=True)
        p.grad = torch.tensor(g, dtype=torch.float64)
        params.append(p)
    total = torch.nn.utils.clip_grad_norm_(params, max_norm)
    ctl = oracle.grad_control(gs, 1.0, max_norm)
    assert not ctl.skip
    assert abs(ctl.norm - float(total)) <= 1e-12 * ctl.norm
    for g, p in zip(gs, params):
        np.testing.assert_allclose(g * ctl.mult, p.grad.numpy(), rtol=1e-13, atol=0)


def test_unscale_by_a_power_of_two_is_exact():
    """A gradient scaler multiplies the loss by S; g*S with inv_loss_scale = 1/S
    gives the unscaled answer exactly (S a power of two)."""
    gs = _grads(2, SHAPES)
    S = 65536.0
    a = oracle.grad_control(gs, 1.0, 0.5)
    b = oracle.grad_control([g * S for g in gs], 1.0 / S, 0.5)
    assert a.norm == b.norm
    for g in gs:
        np.testing.assert_array_equal(g * a.mult, (g * S) * b.mult)


def test_closed_form_norm_of_ones():
    gs = [np.ones((3, 4)), np.ones(10)]
    ctl = oracle.grad_control(gs, 0.5, 0.0)
    assert ctl.norm == pytest.approx(0.5 * math.sqrt(22.0), rel=1e-15)
    assert ctl.mult == 0.5 and not ctl.skip
    clipped = oracle.grad_control(gs, 1.0, 1.0)
    assert clipped.mult == pytest.approx(1.0 / (math.sqrt(22.0) + 1e-6), rel=1e-15)


def test_zero_max_norm_observes_without_clipping():
    gs = _grads(3, SHAPES, 100.0)
    ctl = oracle.grad_control(gs, 1.0, 0.0)
    assert ctl.mult == 1.0
    assert ctl.norm == pytest.approx(math.sqrt(sum(float((g * g).sum()) for g in gs)), rel=1e-14)


def test_norm_below_max_leaves_gradients_alone():
    gs = _grads(4, SHAPES, 1e-3)
    ctl = oracle.grad_control(gs, 1.0, 1.0)
    assert ctl.norm < 1.0 and ctl.mult == 1.0


def test_clip_is_global_across_groups():
    """One factor for every tensor of both groups: the clipped global norm is
    max_norm * norm / (norm + 1e-6); clipping each group on its own would
    leave a different (larger) total."""
    muon = _grads(5, [(8, 8), (4, 16)], 2.0)
    adam = _grads(6, [(100,), (3,)], 0.1)
    max_norm = 1.0
    ctl = oracle.grad_control(muon + adam, 1.0, max_norm)
    clipped = math.sqrt(sum(float(((g * ctl.mult) ** 2).sum()) for g in muon + adam))
    assert clipped == pytest.approx(max_norm * ctl.norm / (ctl.norm + 1e-6), rel=1e-13)
    per_group = [oracle.grad_control(grp, 1.0, max_norm) for grp in (muon, adam)]
    sep = math.sqrt(sum(float(((g * c.mult) ** 2).sum())
                        for grp, c in zip((muon, adam), per_group) for g in grp))
    assert sep > clipped * 1.05


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_non_finite_gradient_skips_the_whole_step(bad):
    gs = _grads(7, SHAPES)
    gs[2][17] = bad
    ctl = oracle.grad_control(gs, 1.0, 1.0)
    assert ctl.skip and ctl.mult == 0.0 and math.isnan(ctl.norm)


def test_large_finite_gradient_is_not_an_overflow():
    gs = _grads(8, SHAPES)
    gs[0][0, 0] = 1e30
    ctl = oracle.grad_control(gs, 1.0, 1.0)
    assert not ctl.skip
    assert ctl.norm == pytest.approx(1e30, rel=1e-12)
    assert ctl.mult == pytest.approx(1e-30, rel=1e-12)
