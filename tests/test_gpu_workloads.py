"""Full-size workloads, run exactly as bench.py runs them (every Muon tensor in
one mh_muon_step_batched call, every AdamW tensor in one mh_adamw_step call),
checked against the fp64 oracle on sampled views and slices that the oracle
can compute one by one (each view's update is independent of the others).

Bars as in test_gpu_muon.py: momentum and AdamW state 1e-6; final parameter
max(1e-3, 2e-2*||dW||/||W||, twice the oracle's own bf16 rounding); NorMuon
state 3e-2.
"""
import gc

import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.helpers import DeviceRun, oracle_adam_tensor, oracle_muon_tensor, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _free(run):
    import torch
    del run
    gc.collect()
    torch.cuda.empty_cache()


def _param_tol(w64, w0, dtype, decay, steps):
    """max(1e-3, the NS bar carried through the total update, the bf16
    rounding floor); over several steps the independent per-step roundings of
    the two runs add like a random walk, hence sqrt(steps)."""
    tol = 1e-3
    dw = w64 - decay ** steps * w0
    tol = max(tol, 2e-2 * np.linalg.norm(dw) / np.linalg.norm(w64))
    if dtype == "bf16":
        tol = max(tol, 2.0 * np.sqrt(steps) * rel_fro(oracle.round_bf16(w64), w64))
    return tol


def _check_muon_views(wl, run, i, views, steps):
    spec = wl.muon[i]
    r, c = spec.rows, spec.cols
    ref = oracle_muon_tensor(wl, i, steps, views=views)
    got_w = to_np(run.mW[i]).reshape(spec.views, r, c)
    got_b = to_np(run.mB[i]).reshape(spec.views, r, c)
    decay = 1 - wl.muon_hp["lr"] * spec.lr_mult * spec.wd
    for k, v in enumerate(views):
        assert rel_fro(got_b[v], ref["B"][k]) < 1e-6, (spec.name, v)
        w0 = W.host_tensor(wl, W.KIND_W, i, offset=v * r * c, count=r * c).reshape(r, c)
        tol = _param_tol(ref["W64"][k], w0, spec.param_dtype, decay, steps)
        err = rel_fro(got_w[v], ref["W"][k])
        assert err < tol, (spec.name, v, err, tol)
        if run.sm[i] is not None:
            got_sm = to_np(run.sm[i]).reshape(spec.views, r)
            assert rel_fro(got_sm[v], ref["sm"][k]) < 3e-2, (spec.name, v)


def _check_adam(wl, run, j, steps, offset=0, count=None):
    spec = wl.adamw[j]
    n = spec.numel if count is None else count
    ref = oracle_adam_tensor(wl, j, steps, offset=offset, count=n)
    sl = slice(offset, offset + n)
    got_w = to_np(run.aW[j].reshape(-1)[sl])
    assert rel_fro(to_np(run.am[j].reshape(-1)[sl]), ref["m"]) < 1e-6
    assert rel_fro(to_np(run.av[j].reshape(-1)[sl]), ref["v"]) < 1e-6
    tol = 1e-6 if spec.param_dtype == "f32" else 1e-3
    assert rel_fro(got_w, ref["W"]) < tol, (spec.name, rel_fro(got_w, ref["W"]))


def _index(wl, name):
    return next(k for k, s in enumerate(wl.muon) if s.name == name)


def test_llama7b_one_step_sampled():
    wl = W.llama7b()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, _index(wl, "l0.q"), [0], 1)
    _check_muon_views(wl, run, _index(wl, "l0.k"), [0], 1)
    _check_muon_views(wl, run, _index(wl, "l31.gate_up"), [1], 1)
    _check_muon_views(wl, run, _index(wl, "l31.down"), [0], 1)
    # AdamW: a 4096-row slice of the embedding and of the head, and a norm.
    _check_adam(wl, run, 0, 1, offset=0, count=4096 * 4096)
    _check_adam(wl, run, 1, 1, offset=124160 * 4096, count=4096 * 4096)
    _check_adam(wl, run, 66, 1)
    _free(run)


def test_gpt124m_ten_steps_sampled():
    wl = W.gpt124m()
    run = DeviceRun(wl)
    for _ in range(wl.steps):
        run.step()
    run.status_ok()
    for name, views in (("l0.q", [0]), ("l0.gate_up", [0, 1]), ("l0.down", [0]),
                        ("l11.v", [0]), ("l11.gate_up", [1])):
        _check_muon_views(wl, run, _index(wl, name), views, wl.steps)
    _check_adam(wl, run, 0, wl.steps, offset=0, count=1 << 20)
    _check_adam(wl, run, 0, wl.steps, offset=50304 * 768 - (1 << 20), count=1 << 20)
    _check_adam(wl, run, 5, wl.steps)
    _free(run)


def test_moe_mla_all_variants_sampled():
    wl = W.moe_mla()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, _index(wl, "e0.gate_up"), [0, 1], 1)
    _check_muon_views(wl, run, _index(wl, "e0.down"), [0], 1)
    _check_muon_views(wl, run, _index(wl, "e63.down"), [0], 1)
    _check_muon_views(wl, run, _index(wl, "mla.kv_b"), list(range(64)), 1)
    _free(run)


def test_single_matrix_config():
    wl = W.single_matrix()
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check_muon_views(wl, run, 0, [0], 1)
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
