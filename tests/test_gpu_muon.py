"""Full Muon step through the C ABI vs the fp64 oracle.

Bars:
* momentum (an fp32 elementwise stage): 1e-6 relative Frobenius;
* the final parameter: 1e-3 relative Frobenius. Where the update is a large
  fraction of the weight (tiny or thin test matrices), the Newton-Schulz bar
  (2e-2 on U) carried through the update, 2e-2 * ||dW|| / ||W||, is the
  larger and is used instead. For bf16 parameters the GPU
  and the oracle each round their own result to bf16, so two results whose
  pre-rounding values differ by a fraction of an ulp can land one ulp apart.
  When the update is only a few bf16 ulps (small test shapes, large weights)
  that rounding noise alone exceeds 1e-3; the bar is then twice the oracle's
  own bf16 quantisation error ||round(W64) - W64|| / ||W64||;
* the update W_new - (1 - lr wd) W_old: 2e-2 relative Frobenius (the
  Newton-Schulz bar) for fp32 parameters, 5e-2 for bf16 parameters (the
  update measured through bf16 storage carries the half-ulp rounding).
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.helpers import DeviceRun, oracle_muon_tensor, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _wl(specs, steps=1, **hp):
    return W.Workload("test", muon=specs, adamw=[], muon_hp=dict(W.MUON_HP, **hp),
                      adam_hp=dict(W.ADAM_HP), steps=steps)


def param_tolerance(w64: np.ndarray, w_prev, dtype: str, decay: float) -> float:
    tol = 1e-3
    if w_prev is not None:
        dw = w64 - decay * w_prev
        tol = max(tol, 2e-2 * np.linalg.norm(dw) / np.linalg.norm(w64))
    if dtype == "bf16":
        tol = max(tol, 2.0 * rel_fro(oracle.round_bf16(w64), w64))
    return tol


def _check(wl, run, tensors=None, w_prev=None):
    for i in (tensors if tensors is not None else range(len(wl.muon))):
        spec = wl.muon[i]
        ref = oracle_muon_tensor(wl, i, run.step_count, keep_unrounded=True)
        shape = (spec.views, spec.rows, spec.cols)
        got_w = to_np(run.mW[i]).reshape(shape)
        got_b = to_np(run.mB[i]).reshape(shape)
        assert rel_fro(got_b, ref["B"]) < 1e-6, (spec.name, rel_fro(got_b, ref["B"]))
        decay = 1 - wl.muon_hp["lr"] * spec.lr_mult * spec.wd
        prev = None if w_prev is None else w_prev[i].reshape(shape)
        tol = param_tolerance(ref["W64"], prev, spec.param_dtype, decay)
        assert rel_fro(got_w, ref["W"]) < tol, (spec.name, rel_fro(got_w, ref["W"]), tol)
        if w_prev is not None:
            decay = 1 - wl.muon_hp["lr"] * spec.lr_mult * spec.wd
            d_got = got_w - decay * w_prev[i].reshape(shape)
            d_ref = ref["W64"] - decay * w_prev[i].reshape(shape)
            if not wl.muon_hp.get("cautious", 0):
                bar = 2e-2 if spec.param_dtype == "f32" else 5e-2
                assert rel_fro(d_got, d_ref) < bar, (spec.name, rel_fro(d_got, d_ref))
        if run.sm[i] is not None:
            # sm averages U^2: a relative error e in U (the NS bar, 2e-2) moves
            # it by up to 2e
            got_sm = to_np(run.sm[i]).reshape(spec.views, spec.rows)
            assert rel_fro(got_sm, ref["sm"]) < 4e-2, (spec.name, rel_fro(got_sm, ref["sm"]))


def test_single_256x1024_fp32():
    wl = W.single_matrix()
    run = DeviceRun(wl)
    W0 = to_np(run.mW[0])
    run.step()
    run.status_ok()
    ref = oracle_muon_tensor(wl, 0, 1)
    got = to_np(run.mW[0])
    assert rel_fro(to_np(run.mB[0]), ref["B"][0]) < 1e-6
    assert rel_fro(got, ref["W"][0]) < 1e-3
    hp = wl.muon_hp
    decay = 1 - hp["lr"] * wl.muon[0].wd
    d_got = got - decay * W0
    d_ref = ref["W"][0] - decay * W0
    assert rel_fro(d_got, d_ref) < 2e-2


MIXED = [W.MuonSpec("sq", 1, 256, 256, "f32", "f32", w_std=1.0, g_std=1.0),
         W.MuonSpec("wide", 1, 200, 456, "bf16", "bf16"),
         W.MuonSpec("tall", 1, 520, 136, "bf16", "f32"),
         W.MuonSpec("views", 2, 384, 128, "bf16", "bf16"),
         W.MuonSpec("ragged", 3, 33, 97, "f32", "bf16", w_std=1.0),
         W.MuonSpec("tiny", 1, 1, 5, "f32", "f32")]


def test_plain_step_mixed_shapes():
    wl = _wl(MIXED)
    run = DeviceRun(wl)
    w0 = [to_np(w) for w in run.mW]
    run.step()
    run.status_ok()
    _check(wl, run, w_prev=w0)


@pytest.mark.parametrize("flags", [dict(normuon=True), dict(muon_plus=True), dict(cautious=1),
                                   dict(cautious=2), dict(nesterov=False),
                                   dict(normuon=True, muon_plus=True, cautious=1),
                                   dict(normuon=True, normuon_eps=1e-4),
                                   dict(shape_rule=1), dict(normuon=True, shape_rule=1, cautious=1)])
def test_variants(flags):
    specs = [W.MuonSpec("a", 2, 256, 512, "f32", "f32", w_std=1.0, g_std=1.0),
             W.MuonSpec("b", 1, 384, 128, "bf16", "bf16"),
             W.MuonSpec("c", 4, 64, 96, "f32", "f32", w_std=0.5, g_std=0.3)]
    wl = _wl(specs, **flags)
    run = DeviceRun(wl)
    w0 = [to_np(w) for w in run.mW]
    run.step()
    run.status_ok()
    _check(wl, run, w_prev=w0)


def test_three_steps_carry_state():
    specs = [W.MuonSpec("a", 1, 256, 640, "f32", "f32", w_std=1.0, g_std=1.0),
             W.MuonSpec("b", 2, 300, 128, "bf16", "bf16")]
    wl = _wl(specs, steps=3, normuon=True, muon_plus=True)
    run = DeviceRun(wl)
    for _ in range(3):
        run.step()
    run.status_ok()
    _check(wl, run)


def test_zero_gradient_is_pure_decay():
    import torch
    specs = [W.MuonSpec("a", 1, 128, 384, "f32", "f32", w_std=1.0)]
    wl = _wl(specs)
    run = DeviceRun(wl)
    run.mG[0].zero_()
    W0 = to_np(run.mW[0])
    run.step()
    torch.cuda.synchronize()
    decay = np.float32(1 - np.float32(0.02) * np.float32(0.01))
    np.testing.assert_allclose(to_np(run.mW[0]), W0 * decay, rtol=1e-6)
    assert torch.all(run.mB[0] == 0)


def test_views_match_separate_tensors():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    r, c = 256, 384
    packed = _wl([W.MuonSpec("p", 2, r, c, "f32", "f32", w_std=1.0, g_std=1.0)])
    run = DeviceRun(packed)
    W0 = run.mW[0].clone()
    G0 = run.mG[0].clone()
    run.step()
    # The same data as two separate tensors.
    Ws = [W0[:r].clone(), W0[r:].clone()]
    Gs = [G0[:r].clone(), G0[r:].clone()]
    Bs = [torch.zeros(r, c, device="cuda") for _ in range(2)]
    ts = [mh.muon_tensor(w, g, b, 1, None, 1.0, 0.01) for w, g, b in zip(Ws, Gs, Bs)]
    ws = torch.empty(mh.muon_workspace_bytes(ts, run.hp), dtype=torch.uint8, device="cuda")
    mh.muon_step_batched(ts, run.hp, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    sep = torch.cat(Ws)
    assert rel_fro(to_np(run.mW[0]), to_np(sep)) < 1e-6


def test_repeat_call_same_workspace_is_reproducible():
    import torch
    specs = [W.MuonSpec("a", 1, 256, 512, "f32", "f32", w_std=1.0, g_std=1.0)]
    wl = _wl(specs)
    r1, r2 = DeviceRun(wl), DeviceRun(wl)
    r1.step()
    r2.ws.fill_(0xAB)  # stale workspace contents must not matter
    r2.step()
    torch.cuda.synchronize()
    assert rel_fro(to_np(r1.mW[0]), to_np(r2.mW[0])) < 1e-6


def test_polar_express_schedule_step():
    """flaxchat "Muon Algorithm" step 2 in the full step: X = Q / (||Q|| * 1.01),
    one (a, b, c) per iteration (arbitrary values: the page prints none)."""
    sched = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.6, -2.4, 0.8), (2.0, -1.5, 0.5),
             (1.875, -1.25, 0.375)]
    specs = [W.MuonSpec("a", 2, 256, 512, "f32", "f32", w_std=1.0, g_std=1.0),
             W.MuonSpec("b", 1, 384, 128, "bf16", "bf16"),
             W.MuonSpec("c", 1, 96, 200, "f32", "f32", w_std=0.5, g_std=0.3)]
    wl = _wl(specs, coeffs=sched, eps=0.0, norm_scale=1.01)
    run = DeviceRun(wl)
    w0 = [to_np(w).copy() for w in run.mW]
    run.step()
    run.status_ok()
    _check(wl, run, w_prev=w0)
