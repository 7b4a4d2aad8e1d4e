"""Full Muon step through the C ABI vs the fp64 oracle.

Bars (tests.parity, applied by tests.helpers.check_muon_views):
* momentum (an fp32 elementwise stage): element by element,
  |got - want| <= 1e-6 |want| + 2 atol, atol the running bound on the
  kernel's fp32 rounding;
* fp32 parameters: the update W_new - base (base = the decayed previous
  weight, or the previous weight under a cautious mask) within 2e-2 (the
  Newton-Schulz bar) of the oracle's, relative Frobenius; the parameter
  within 1e-3 unless the update is a large part of it (then the
  Newton-Schulz bar carried through); no systematic update scale error
  above 1 %;
* bf16 parameters: every element at most one bf16 spacing (plus ten times
  the per-element size of the Newton-Schulz bar, for values near zero) from
  the oracle's rounded value; the fraction of elements one spacing away, and
  the update's relative error, within 1.25x of what the Newton-Schulz bar
  predicts through the rounding; no systematic update scale error above 1 %;
* NorMuon state: 4e-2 relative Frobenius (it averages U^2, so a relative
  error e in U moves it by up to 2e: twice the Newton-Schulz bar).
Several steps are checked one step at a time from the device's own state
before the last step, plus the momentum over the whole run.
"""
import numpy as np
import pytest

from synth import workloads as W
from tests.helpers import (DeviceRun, check_muon_views, oracle_muon_step_from,
                           oracle_muon_tensor, rel_fro, to_np)
from tests.parity import check_fp32

pytestmark = pytest.mark.gpu


def _wl(specs, steps=1, **hp):
    return W.Workload("test", muon=specs, adamw=[], muon_hp=dict(W.MUON_HP, **hp),
                      adam_hp=dict(W.ADAM_HP), steps=steps)


def snapshot(run, i):
    """The device's W, B and NorMuon state of Muon tensor i, as (views, r, c)."""
    spec = run.wl.muon[i]
    shape = (spec.views, spec.rows, spec.cols)
    sm = None if run.sm[i] is None else to_np(run.sm[i]).reshape(spec.views, spec.rows)
    return to_np(run.mW[i]).reshape(shape), to_np(run.mB[i]).reshape(shape), sm


def _check(wl, run, tensors=None):
    """Parity of a run that has taken one step from the workload's initial state."""
    assert run.step_count == 1
    for i in (tensors if tensors is not None else range(len(wl.muon))):
        ref = oracle_muon_tensor(wl, i, 1)
        got_w, got_b, got_sm = snapshot(run, i)
        check_muon_views(wl, i, ref, got_w, got_b, got_sm)


def _run_and_check_last_step(wl, run, steps):
    """Runs ``steps`` steps; checks the last one from the device's state before
    it, and the momentum over the whole run."""
    for _ in range(steps - 1):
        run.step()
    before = [snapshot(run, i) for i in range(len(wl.muon))]
    run.step()
    run.status_ok()
    for i, spec in enumerate(wl.muon):
        views = list(range(spec.views))
        w0, b0, sm0 = before[i]
        ref = oracle_muon_step_from(wl, i, steps - 1, views, w0, b0, sm0)
        got_w, got_b, got_sm = snapshot(run, i)
        check_muon_views(wl, i, ref, got_w, got_b, got_sm, what=f"{wl.name} step {steps}")
        traj = oracle_muon_tensor(wl, i, steps)
        for k in views:
            check_fp32(got_b[k], traj["B"][k], traj["B_atol"][k],
                       f"{spec.name}[{k}] momentum over {steps} steps")


def test_single_256x1024_fp32():
    wl = W.single_matrix()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check(wl, run)


MIXED = [W.MuonSpec("sq", 1, 256, 256, "f32", "f32", w_std=1.0, g_std=1.0),
         W.MuonSpec("wide", 1, 200, 456, "bf16", "bf16"),
         W.MuonSpec("tall", 1, 520, 136, "bf16", "f32"),
         W.MuonSpec("views", 2, 384, 128, "bf16", "bf16"),
         W.MuonSpec("ragged", 3, 33, 97, "f32", "bf16", w_std=1.0),
         W.MuonSpec("tiny", 1, 1, 5, "f32", "f32")]


def test_plain_step_mixed_shapes():
    wl = _wl(MIXED)
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check(wl, run)


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
    run.step()
    run.status_ok()
    _check(wl, run)


def test_three_steps_carry_state():
    specs = [W.MuonSpec("a", 1, 256, 640, "f32", "f32", w_std=1.0, g_std=1.0),
             W.MuonSpec("b", 2, 300, 128, "bf16", "bf16")]
    wl = _wl(specs, steps=3, normuon=True, muon_plus=True)
    _run_and_check_last_step(wl, DeviceRun(wl), 3)


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
    run.step()
    run.status_ok()
    _check(wl, run)
