"""Newton-Schulz through the C ABI (grouped tcgen05 GEMMs) vs the fp64 oracle.

Bar: bf16-operand NS output within 2e-2 relative Frobenius error. Single-step
runs with special coefficients isolate the three GEMM stages and the folded
normalisation, with tighter bounds (they involve fewer bf16 roundings).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import rel_fro, to_np

pytestmark = pytest.mark.gpu

COEFFS = (3.4445, -4.7750, 2.0315)


def gpu_ns(mats, steps=5, coeffs=COEFFS, eps=1e-7, views=None, in_dtype="f32", out_dtype="f32",
           norm_scale=1.0):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    xs = [torch.tensor(m.reshape(-1, m.shape[-1]), dtype=tdt[in_dtype], device="cuda") for m in mats]
    outs = [torch.full_like(x, float("nan"), dtype=tdt[out_dtype]) for x in xs]
    mh.newton_schulz(xs, outs, views=views, steps=steps, coeffs=coeffs, eps=eps,
                     norm_scale=norm_scale)
    torch.cuda.synchronize()
    return [to_np(o) for o in outs]


def _mat(seed, tid, shape, std=1.0):
    return synth.normal(seed, tid, shape, std=std).astype(np.float64)


SHAPES = [(128, 512), (512, 128), (256, 256), (300, 700), (700, 300), (1, 64), (64, 1),
          (130, 136), (8, 8), (384, 1536), (1000, 1000), (1024, 4096)]


@pytest.mark.parametrize("shape", SHAPES)
def test_ns_matches_oracle(shape):
    Q = _mat(11, shape[0] * 7 + shape[1], shape)
    got = gpu_ns([Q])[0]
    want = oracle.newton_schulz(Q)
    assert np.all(np.isfinite(got))
    assert rel_fro(got, want) < 2e-2, rel_fro(got, want)


def test_ns_mixed_classes_one_call():
    shapes = [(256, 1024), (1024, 256), (200, 300), (768, 768), (128, 512), (256, 1024)]
    mats = [_mat(12, i, s) for i, s in enumerate(shapes)]
    gots = gpu_ns(mats)
    for Q, got in zip(mats, gots):
        assert rel_fro(got, oracle.newton_schulz(Q)) < 2e-2


def test_ns_views_are_independent():
    k, r, c = 3, 96, 160
    Q = _mat(13, 1, (k * r, c))
    got = gpu_ns([Q], views=[k])[0].reshape(k, r, c)
    for v in range(k):
        assert rel_fro(got[v], oracle.newton_schulz(Q[v * r:(v + 1) * r])) < 2e-2


def test_ns_more_than_eight_classes():
    shapes = [(64 + 16 * i, 96 + 32 * i) for i in range(11)]
    mats = [_mat(14, i, s) for i, s in enumerate(shapes)]
    for Q, got in zip(mats, gpu_ns(mats)):
        assert rel_fro(got, oracle.newton_schulz(Q)) < 2e-2


@pytest.mark.parametrize("shape", [(256, 768), (768, 256), (200, 328)])
def test_stage_normalisation_only(shape):
    # (a, b, c) = (1, 0, 0), one step: U = Q / (||Q|| + eps); only the bf16
    # rounding of Q and of U remain.
    Q = _mat(15, 1, shape, std=3.0)
    got = gpu_ns([Q], steps=1, coeffs=(1.0, 0.0, 0.0))[0]
    assert rel_fro(got, oracle.newton_schulz(Q, steps=1, coeffs=(1.0, 0.0, 0.0))) < 5e-3


@pytest.mark.parametrize("shape", [(256, 768), (768, 256), (300, 200), (640, 640)])
def test_stage_gram_and_apply(shape):
    # (0, 1, 0): U = (X X^T) X -- checks the gram, its mirrored upper-triangle
    # store and the MN-major apply.
    Q = _mat(16, 2, shape)
    got = gpu_ns([Q], steps=1, coeffs=(0.0, 1.0, 0.0))[0]
    assert rel_fro(got, oracle.newton_schulz(Q, steps=1, coeffs=(0.0, 1.0, 0.0))) < 1e-2


@pytest.mark.parametrize("shape", [(256, 768), (300, 200), (640, 640)])
def test_stage_poly(shape):
    # (0, 0, 1): U = (X X^T)^2 X -- checks the A A product of the poly stage.
    Q = _mat(17, 3, shape)
    got = gpu_ns([Q], steps=1, coeffs=(0.0, 0.0, 1.0))[0]
    assert rel_fro(got, oracle.newton_schulz(Q, steps=1, coeffs=(0.0, 0.0, 1.0))) < 1e-2


def test_zero_steps_is_normalisation():
    Q = _mat(18, 1, (100, 260), std=5.0)
    got = gpu_ns([Q], steps=0)[0]
    assert rel_fro(got, Q / (np.linalg.norm(Q) + 1e-7)) < 5e-3


def test_zero_matrix_stays_zero():
    got = gpu_ns([np.zeros((128, 384)), np.zeros((300, 100))])
    for g in got:
        assert np.all(g == 0)


def test_tall_equals_transpose_of_wide():
    Q = _mat(19, 1, (200, 520))
    wide, tall = gpu_ns([Q, Q.T.copy()])
    np.testing.assert_allclose(tall, wide.T, rtol=0, atol=1e-6)


def test_bf16_input_and_output():
    Q = synth.normal(20, 1, (512, 1024), dtype="bf16").astype(np.float64)
    got = gpu_ns([Q], in_dtype="bf16", out_dtype="bf16")[0]
    assert rel_fro(got, oracle.newton_schulz(Q)) < 2e-2


def test_singular_values_in_quintic_band():
    Q = _mat(21, 1, (512, 2048))
    got = gpu_ns([Q])[0]
    sv = np.linalg.svd(got, compute_uv=False)
    assert sv.min() > 0.6 and sv.max() < 1.3


@pytest.mark.parametrize("shape", [(2048, 8192), (4096, 4096)])
def test_ns_large(shape):
    Q = _mat(22, shape[0], shape)
    got = gpu_ns([Q])[0]
    assert rel_fro(got, oracle.newton_schulz(Q)) < 2e-2


# ---- coefficient schedules and the Polar Express normalisation (flaxchat "Muon
# Algorithm" step 2). The page prints no coefficients; any schedule must match.
SCHED = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.6, -2.4, 0.8), (2.0, -1.5, 0.5),
         (1.875, -1.25, 0.375)]


@pytest.mark.parametrize("shape", [(256, 768), (768, 256), (300, 200), (64, 1000)])
@pytest.mark.parametrize("norm_scale,eps", [(1.01, 0.0), (1.0, 1e-7)])
def test_schedule_matches_oracle(shape, norm_scale, eps):
    Q = _mat(40, shape[0] + shape[1], shape)
    got = gpu_ns([Q], steps=5, coeffs=SCHED, eps=eps, norm_scale=norm_scale)[0]
    want = oracle.newton_schulz(Q, steps=5, coeffs=SCHED, eps=eps, norm_scale=norm_scale)
    assert rel_fro(got, want) < 2e-2, rel_fro(got, want)
    # a constant schedule is the plain iteration
    const = gpu_ns([Q], steps=5, coeffs=[COEFFS] * 5)[0]
    assert rel_fro(const, gpu_ns([Q])[0]) < 1e-6


def test_schedule_zero_matrix_without_eps_stays_zero():
    got = gpu_ns([np.zeros((128, 384)), np.zeros((300, 100))], steps=5, coeffs=SCHED, eps=0.0,
                 norm_scale=1.01)
    for g in got:
        assert np.all(g == 0)


def test_zero_steps_with_norm_scale():
    Q = _mat(41, 1, (100, 260), std=5.0)
    got = gpu_ns([Q], steps=0, coeffs=[], eps=0.0, norm_scale=1.01)[0]
    assert rel_fro(got, Q / (np.linalg.norm(Q) * 1.01)) < 5e-3
