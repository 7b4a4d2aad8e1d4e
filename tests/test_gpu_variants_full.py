"""The 7B-shape set with the optional rows switched on, run exactly as
bench.py runs it (bench.DeviceWorkload: every Muon tensor in one call, every
AdamW tensor in one call), checked on sampled views and slices against the
oracle.

* bf16 optimizer state with stochastic rounding (dew.training.optim,
  "bf16_moments", "stochastic_round_bf16"): momentum and Adam moments bit for
  bit wherever a few-ulp fp32 difference cannot move the rounding (see
  tests/test_gpu_sr.py), parameters to the final-parameter bar with > 85 %
  of their rounding decisions equal to the oracle's (the NS error moves a
  few per cent; a wrong key would leave about two thirds).
* gradient control (kimi-k3 "Optimization", "Keep the arithmetic and
  gradients under control"): the global norm of all 8.03 G gradient elements
  against torch's float64 norm on the device, and the clipped step on sampled
  views against the oracle run on the clipped gradients.
"""
import numpy as np
import pytest

import bench
import oracle
from synth import workloads as W
from tests.helpers import oracle_hparams, rel_fro, to_np
from tests.test_gpu_sr import _check_state, _expected_bits

pytestmark = pytest.mark.gpu


def _index(wl, name):
    return next(k for k, s in enumerate(wl.muon) if s.name == name)


def _views(wl, i, views, mult=1.0):
    spec = wl.muon[i]
    r, c = spec.rows, spec.cols
    out = []
    for v in views:
        off, cnt = v * r * c, r * c
        w = W.host_tensor(wl, W.KIND_W, i, offset=off, count=cnt).reshape(r, c)
        g = W.host_tensor(wl, W.KIND_G, i, offset=off, count=cnt).reshape(r, c)
        out.append((v, w, g, oracle.muon_step_view(w, mult * g, np.zeros((r, c)),
                                                   oracle_hparams(wl), spec.lr_mult, spec.wd)))
    return out


def _free(dw):
    import gc
    import torch
    del dw
    gc.collect()
    torch.cuda.empty_cache()


def test_llama7b_bf16_state_one_step_sampled():
    import torch
    wl = W.llama7b_bf16_state()
    dw = bench.DeviceWorkload(wl, torch.device("cuda", 0))
    stream = torch.cuda.current_stream()
    dw.step(stream)
    torch.cuda.synchronize()
    dw.check_status(stream)
    seed = dw.step_count
    agree = total = 0
    for name, views in (("l0.q", [0]), ("l31.gate_up", [1]), ("l17.down", [0])):
        i = _index(wl, name)
        spec = wl.muon[i]
        r, c = spec.rows, spec.cols
        gotB = dw.mB[i].reshape(spec.views, r, c)
        gotW = dw.mW[i].reshape(spec.views, r, c)
        for v, w, g, ref in _views(wl, i, views):
            off = v * r * c
            # momentum from zero: B = (1 - mu) G, rounded stochastically
            want, amb = _expected_bits(ref.B, seed, oracle.sr_stream(i, oracle.MOMENT_FIRST),
                                       terms=np.abs(0.05 * g), index0=off)
            got = gotB[v].contiguous().view(torch.int16).cpu().numpy().astype(np.uint16).ravel()
            assert np.all(got[~amb] == want[~amb]), name
            tol = max(1e-3, 2e-2 * np.linalg.norm(ref.W - 0.9998 * w) / np.linalg.norm(ref.W),
                      2.0 * rel_fro(oracle.round_bf16(ref.W), ref.W))
            assert rel_fro(to_np(gotW[v]), ref.W) < 1.5 * tol, name
            wbits, _ = _expected_bits(ref.W, seed, oracle.sr_stream(i, oracle.MOMENT_PARAM),
                                      index0=off)
            gw = gotW[v].contiguous().view(torch.int16).cpu().numpy().astype(np.uint16).ravel()
            agree += int(np.sum(gw == wbits))
            total += gw.size
    # The update here is a few bf16 spacings of the weights (std 0.02), so the
    # NS error moves a few per cent of the decisions; a wrong key, stream or
    # index would agree on about two thirds.
    assert agree / total > 0.85, agree / total
    # AdamW: a 4096-row slice of the embedding (bias-corrected step 1)
    n = 4096 * 4096
    hp = wl.adam_hp
    w = W.host_tensor(wl, W.KIND_AW, 0, count=n)
    g = W.host_tensor(wl, W.KIND_AG, 0, count=n)
    Wn, M, V = oracle.adamw_step(w, g, np.zeros(n), np.zeros(n), hp["lr"], hp["betas"][0],
                                 hp["betas"][1], hp["eps"], wl.adamw[0].wd, 1)
    _check_state(dw.am[0].reshape(-1)[:n], M, 1, oracle.sr_stream(0, oracle.MOMENT_FIRST), "m",
                 terms=np.abs(0.1 * g))
    _check_state(dw.av[0].reshape(-1)[:n], V, 1, oracle.sr_stream(0, oracle.MOMENT_SECOND), "v",
                 terms=np.abs(0.05 * g * g))
    _check_state(dw.aW[0].reshape(-1)[:n], Wn, 1, oracle.sr_stream(0, oracle.MOMENT_PARAM), "W",
                 terms=np.abs(w) + 10.0 * np.abs(Wn - w))
    _free(dw)


def test_llama7b_clipped_step_sampled():
    import torch
    wl = W.llama7b()
    max_norm = 10.0
    dw = bench.DeviceWorkload(wl, torch.device("cuda", 0), max_grad_norm=max_norm)
    stream = torch.cuda.current_stream()
    norm64 = torch.sqrt(sum(torch.sum(g.double() ** 2) for g in dw.mG + dw.aG)).item()
    dw.step(stream)
    torch.cuda.synchronize()
    dw.check_status(stream)
    ctl = dw.control
    assert int(ctl.skip.item()) == 0 and int(ctl.step.item()) == 1
    assert abs(float(ctl.norm.item()) - norm64) <= 1e-6 * norm64
    mult = min(1.0, max_norm / (norm64 + 1e-6))
    assert mult < 0.5                                  # clipping is active
    assert abs(float(ctl.grad_mult.item()) - mult) <= 1e-6 * mult
    for name, views in (("l3.o", [0]), ("l30.gate_up", [0])):
        i = _index(wl, name)
        spec = wl.muon[i]
        r, c = spec.rows, spec.cols
        gotB = to_np(dw.mB[i]).reshape(spec.views, r, c)
        gotW = to_np(dw.mW[i]).reshape(spec.views, r, c)
        for v, w, g, ref in _views(wl, i, views, mult):
            assert rel_fro(gotB[v], ref.B) < 1e-6, name
            tol = max(1e-3, 2e-2 * np.linalg.norm(ref.W - 0.9998 * w) / np.linalg.norm(ref.W),
                      2.0 * rel_fro(oracle.round_bf16(ref.W), ref.W))
            assert rel_fro(gotW[v], oracle.round_bf16(ref.W)) < tol, name
    n = 1 << 22
    hp = wl.adam_hp
    w = W.host_tensor(wl, W.KIND_AW, 1, count=n)
    g = W.host_tensor(wl, W.KIND_AG, 1, count=n)
    Wn, M, V = oracle.adamw_step(w, mult * g, np.zeros(n), np.zeros(n), hp["lr"],
                                 hp["betas"][0], hp["betas"][1], hp["eps"], wl.adamw[1].wd, 1)
    assert rel_fro(to_np(dw.am[1].reshape(-1)[:n]), M) < 1e-6
    assert rel_fro(to_np(dw.av[1].reshape(-1)[:n]), V) < 1e-6
    assert rel_fro(to_np(dw.aW[1].reshape(-1)[:n]), oracle.round_bf16(Wn)) < 1e-3
    _free(dw)
