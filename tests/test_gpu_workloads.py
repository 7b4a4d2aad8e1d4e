"""Full-size workloads, run exactly as bench.py runs them (every Muon tensor in
one mh_muon_step_batched call, every AdamW tensor in one mh_adamw_step call),
checked against the fp64 oracle on sampled views and slices that the oracle
can compute one by one (each view's update is independent of the others).

Bars as in test_gpu_muon.py and test_gpu_adamw.py (tests.parity): momentum,
AdamW moments and fp32 AdamW parameters element by element against the
running bound on the kernels' fp32 rounding; parameters after a Muon step by
the update they received (fp32: the Newton-Schulz bar; bf16: one spacing
from the oracle's rounded value, the flip rate and the update error the
Newton-Schulz bar predicts through the rounding, no systematic scale error);
NorMuon state 3e-2. The ten-step 124M run is checked on its last step from
the device's own state before it, on the momentum over all ten steps, and on
the parameter's drift over the run.
"""
import gc

import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.helpers import (DeviceRun, check_adam_result, check_muon_views, oracle_adam_step_from,
                           oracle_adam_tensor, oracle_muon_step_from, oracle_muon_tensor, rel_fro,
                           to_np)
from tests.parity import check_fp32, record

pytestmark = pytest.mark.gpu


def _free(run):
    import torch
    del run
    gc.collect()
    torch.cuda.empty_cache()


def _device_views(run, i, views):
    spec = run.wl.muon[i]
    shape = (spec.views, spec.rows, spec.cols)
    w = to_np(run.mW[i]).reshape(shape)[views]
    b = to_np(run.mB[i]).reshape(shape)[views]
    sm = None if run.sm[i] is None else to_np(run.sm[i]).reshape(spec.views, spec.rows)[views]
    return w, b, sm


def _check_muon_views(wl, run, i, views, sm_bar=3e-2):
    """One step from the workload's initial state."""
    ref = oracle_muon_tensor(wl, i, 1, views=views)
    w, b, sm = _device_views(run, i, views)
    check_muon_views(wl, i, ref, w, b, sm, sm_bar=sm_bar)


def _drift_tol(w64, w0, dtype, decay, steps):
    """Bar on a parameter's distance from the oracle's after ``steps`` steps
    run independently on both sides: max(1e-3, the Newton-Schulz bar carried
    through the total update, and for bf16 twice the oracle's own rounding
    error times sqrt(steps)). Each step's roundings can land one spacing
    apart on the two sides (the flip rate the one-step checks measure), and
    a plain Muon or AdamW update does not depend on the weight, so those
    differences persist and add up like a random walk."""
    tol = max(1e-3, 2e-2 * np.linalg.norm(w64 - decay ** steps * w0) / np.linalg.norm(w64))
    if dtype == "bf16":
        tol = max(tol, 2.0 * np.sqrt(steps) * rel_fro(oracle.round_bf16(w64), w64))
    return tol


def _adam_slice(run, j, offset, n):
    sl = slice(offset, offset + n)
    return (to_np(run.aW[j].reshape(-1)[sl]), to_np(run.am[j].reshape(-1)[sl]),
            to_np(run.av[j].reshape(-1)[sl]))


def _check_adam(wl, run, j, steps, offset=0, count=None):
    """A slice of AdamW tensor j after ``steps`` steps from the initial state."""
    spec = wl.adamw[j]
    n = spec.numel if count is None else count
    ref = oracle_adam_tensor(wl, j, steps, offset=offset, count=n)
    check_adam_result(*_adam_slice(run, j, offset, n), ref, spec.param_dtype,
                      f"{wl.name}:{spec.name}[{offset}:{offset + n}]", steps=steps)


def _index(wl, name):
    return next(k for k, s in enumerate(wl.muon) if s.name == name)


def test_llama7b_one_step_sampled():
    wl = W.llama7b()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, _index(wl, "l0.q"), [0])
    _check_muon_views(wl, run, _index(wl, "l0.k"), [0])
    _check_muon_views(wl, run, _index(wl, "l31.gate_up"), [1])
    _check_muon_views(wl, run, _index(wl, "l31.down"), [0])
    # AdamW: a 4096-row slice of the embedding and of the head, and a norm.
    _check_adam(wl, run, 0, 1, offset=0, count=4096 * 4096)
    _check_adam(wl, run, 1, 1, offset=124160 * 4096, count=4096 * 4096)
    _check_adam(wl, run, 66, 1)
    _free(run)


def test_gpt124m_ten_steps_sampled():
    wl = W.gpt124m()
    run = DeviceRun(wl)
    sample = (("l0.q", [0]), ("l0.gate_up", [0, 1]), ("l0.down", [0]), ("l11.v", [0]),
              ("l11.gate_up", [1]))
    adam_sample = ((0, 0, 1 << 20), (0, 50304 * 768 - (1 << 20), 1 << 20), (5, 0, 768))
    for _ in range(wl.steps - 1):
        run.step()
    before = {name: _device_views(run, _index(wl, name), views) for name, views in sample}
    before_adam = {a: _adam_slice(run, *a) for a in adam_sample}
    run.step()
    run.status_ok()
    for name, views in sample:
        i = _index(wl, name)
        spec = wl.muon[i]
        w0, b0, sm0 = before[name]
        # the last step, from the device's own state before it
        ref = oracle_muon_step_from(wl, i, wl.steps - 1, views, w0, b0, sm0)
        w, b, sm = _device_views(run, i, views)
        check_muon_views(wl, i, ref, w, b, sm, what=f"{wl.name} step {wl.steps}")
        # the whole run: momentum element by element, the parameter's drift
        traj = oracle_muon_tensor(wl, i, wl.steps, views=views)
        decay = 1 - wl.muon_hp["lr"] * spec.lr_mult * spec.wd
        r, c = spec.rows, spec.cols
        for k, v in enumerate(views):
            check_fp32(b[k], traj["B"][k], traj["B_atol"][k],
                       f"{wl.name}:{name}[{v}] momentum over {wl.steps} steps")
            w_init = W.host_tensor(wl, W.KIND_W, i, offset=v * r * c, count=r * c).reshape(r, c)
            tol = _drift_tol(traj["W64"][k], w_init, spec.param_dtype, decay, wl.steps)
            err = rel_fro(w[k], traj["W"][k])
            record("drift", f"{wl.name}:{name}[{v}] over {wl.steps} steps", w_rel=err, bar=tol)
            assert err < tol, (name, v, err, tol)
    for j, off, n in adam_sample:
        # the last step from the device's own state, then the whole run
        ref = oracle_adam_step_from(wl, j, wl.steps - 1, off, n, *before_adam[(j, off, n)])
        check_adam_result(*_adam_slice(run, j, off, n), ref, wl.adamw[j].param_dtype,
                          f"{wl.name}:{wl.adamw[j].name}[{off}:{off + n}] step {wl.steps}")
        _check_adam(wl, run, j, wl.steps, offset=off, count=n)
    _free(run)


def test_moe_mla_all_variants_sampled():
    wl = W.moe_mla()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, _index(wl, "e0.gate_up"), [0, 1])
    _check_muon_views(wl, run, _index(wl, "e0.down"), [0])
    _check_muon_views(wl, run, _index(wl, "e63.down"), [0])
    _check_muon_views(wl, run, _index(wl, "mla.kv_b"), list(range(64)))
    _free(run)


def test_single_matrix_config():
    wl = W.single_matrix()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, 0, [0])
    _free(run)


def test_adamw_2p30_fp32_sampled():
    wl = W.adamw_2p30()
    run = DeviceRun(wl)
    run.step()
    n = 1 << 30
    for off in (0, n // 2 + 12345, n - (1 << 20)):
        _check_adam(wl, run, 0, 1, offset=off, count=1 << 20)
    _free(run)


@pytest.mark.parametrize("aspect,n,batch,views", [("4:1", 2048, 4, [0, 3]),
                                                   ("1:4", 1024, 16, [0, 15]),
                                                   ("1:1", 4096, 4, [2])])
def test_ns_sweep_points_sampled(aspect, n, batch, views):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    import synth
    from synth.gpu import fill_normal
    r, c = {"1:1": (n, n), "1:4": (n, 4 * n), "4:1": (4 * n, n)}[aspect]
    x = torch.empty(batch * r, c, dtype=torch.bfloat16, device="cuda")
    fill_normal(x, 0, 5000 + n, 1.0)   # the tensor bench.py --workload ns uses
    out = torch.empty_like(x)
    mh.newton_schulz([x], [out], views=[batch])
    torch.cuda.synchronize()
    got = out.view(batch, r, c)
    for v in views:
        q = synth.normal(0, 5000 + n, (r, c), dtype="bf16", offset=v * r * c).astype(np.float64)
        err = rel_fro(to_np(got[v]), oracle.newton_schulz(q))
        assert err < 2e-2, (aspect, n, v, err)
