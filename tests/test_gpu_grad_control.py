"""Gradient control on the GPU against the oracle: global norm, clip factor,
overflow skip, and whole hybrid steps run under it.

kimi-k3 "Optimization", "Keep the arithmetic and gradients under control";
dew.training.optim "build_optimizer" (the clip reads every gradient of every
group together).

Bars: norm and factor 1e-6 relative (fp32 squares summed in fp64 partials);
skip and step count exact; after steps under clipping the momentum, the AdamW
moments and the fp32 AdamW parameters element by element against the running
bound on fp32 rounding (tests.parity; the clip factor adds four fp32 unit
roundoffs to every gradient: its own rounding, the norm's, and the product),
Muon parameters within the final-parameter bar (max(1e-3, 2e-2 * ||dW|| /
||W||)) over the run.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from tests.helpers import rel_fro, to_np
from tests.parity import U32, adamw_atol, check_fp32, momentum_atol

G_REL = 4 * U32   # relative error of a clipped gradient on the device

pytestmark = pytest.mark.gpu

MUON = [("q", (256, 256), 1, "bf16"), ("gate_up", (2 * 384, 128), 2, "f32"),
        ("down", (128, 384), 1, "f32")]
ADAM = [("embed", (1000, 64), "f32"), ("norm", (64,), "bf16"), ("odd", (4099,), "f32")]
HP = oracle.MuonHparams(lr=0.02, momentum=0.95, nesterov=True)
ADAM_HP = dict(lr=3e-4, betas=(0.9, 0.95), eps=1e-8)
MUON_WD, ADAM_WD = 0.01, 0.1


def _host_grad(seed, idx, shape, dtype, scale=1.0):
    return synth.normal(40 + seed, idx, shape, std=1e-3 * scale, dtype=dtype).astype(np.float64)


def _dev(x, dtype):
    import torch
    t = torch.tensor(np.asarray(x), dtype=torch.float64, device="cuda")
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


def _grads(step, scale=1.0):
    hm = [_host_grad(step, i, s, d, scale) for i, (_, s, _, d) in enumerate(MUON)]
    ha = [_host_grad(step, 10 + i, s, d, scale) for i, (_, s, d) in enumerate(ADAM)]
    return hm, ha


def _control(grads_dev, inv=1.0, max_norm=0.0, ctl=None):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    ctl = ctl or mh.GradientControl("cuda")
    mh.grad_prepare(grads_dev, ctl, inv, max_norm)
    torch.cuda.synchronize()
    return ctl


@pytest.mark.parametrize("inv,max_frac", [(1.0, 0.0), (1.0, 0.4), (1.0, 3.0), (1.0 / 256, 0.4)])
def test_prepare_matches_oracle(inv, max_frac):
    hm, ha = _grads(0, 1.0 / inv)
    host = hm + ha
    dtypes = [d for *_, d in MUON] + [d for *_, d in ADAM]
    dev = [_dev(g, d) for g, d in zip(host, dtypes)]
    # a 16-byte-misaligned gradient and ragged lengths take the scalar path
    odd = synth.normal(99, 1, (70001,), std=1e-3 / inv).astype(np.float32).astype(np.float64)
    import torch
    big = torch.tensor(np.concatenate([[0.0], odd]), dtype=torch.float32, device="cuda")
    dev.append(big[1:])
    host.append(odd)
    norm0 = math.sqrt(sum(float(np.dot((g * inv).ravel(), (g * inv).ravel())) for g in host))
    max_norm = max_frac * norm0
    ref = oracle.grad_control(host, inv, max_norm)
    ctl = _control(dev, inv, max_norm)
    assert int(ctl.skip.item()) == 0
    assert int(ctl.step.item()) == 1
    assert abs(float(ctl.norm.item()) - ref.norm) <= 1e-6 * ref.norm
    assert abs(float(ctl.grad_mult.item()) - ref.mult) <= 1e-6 * ref.mult


@pytest.mark.parametrize("bad_at", [0, 3])
def test_non_finite_gradient_sets_skip(bad_at):
    hm, ha = _grads(1)
    dtypes = [d for *_, d in MUON] + [d for *_, d in ADAM]
    dev = [_dev(g, d) for g, d in zip(hm + ha, dtypes)]
    dev[bad_at].view(-1)[123] = float("nan") if bad_at else float("inf")
    ctl = _control(dev, 1.0, 1.0)
    assert int(ctl.skip.item()) == 1
    assert float(ctl.grad_mult.item()) == 0.0
    assert math.isnan(float(ctl.norm.item()))
    assert int(ctl.step.item()) == 0


def test_norm_without_clipping_and_empty_list():
    hm, ha = _grads(2)
    dtypes = [d for *_, d in MUON] + [d for *_, d in ADAM]
    dev = [_dev(g, d) for g, d in zip(hm + ha, dtypes)]
    ref = oracle.grad_control(hm + ha, 0.5, 0.0)
    ctl = _control(dev, 0.5, 0.0)
    assert float(ctl.grad_mult.item()) == 0.5
    assert abs(float(ctl.norm.item()) - ref.norm) <= 1e-6 * ref.norm
    empty = _control([], 0.25, 1.0)
    assert float(empty.norm.item()) == 0.0 and float(empty.grad_mult.item()) == 0.25
    assert int(empty.skip.item()) == 0


def test_huge_finite_gradient_gives_zero_factor_not_skip():
    """The fp32 squares of |u| > 1.8e19 overflow: the norm is inf and the
    factor 0 (the oracle's fp64 factor is 1e-30 * max_norm); never a skip."""
    import torch
    g = torch.zeros(1000, dtype=torch.float32, device="cuda")
    g[7] = 1e30
    ctl = _control([g], 1.0, 1.0)
    assert int(ctl.skip.item()) == 0
    assert math.isinf(float(ctl.norm.item()))
    assert float(ctl.grad_mult.item()) == 0.0
    assert not oracle.grad_control([to_np(g)], 1.0, 1.0).skip


def test_prepare_is_bitwise_reproducible():
    hm, ha = _grads(3)
    dtypes = [d for *_, d in MUON] + [d for *_, d in ADAM]
    dev = [_dev(g, d) for g, d in zip(hm + ha, dtypes)]
    a = _control(dev, 1.0, 0.1)
    b = _control(dev, 1.0, 0.1)
    assert a.norm.item() == b.norm.item() and a.grad_mult.item() == b.grad_mult.item()


def _oracle_run(steps_grads, max_norm, inv):
    """The oracle's hybrid steps under gradient control (skipped steps change
    nothing and do not advance AdamW's step count)."""
    W_m = [synth.normal(7, i, s, std=0.02).astype(np.float32).astype(np.float64)
           for i, (_, s, _, _) in enumerate(MUON)]
    B_m = [np.zeros(s) for _, s, _, _ in MUON]
    W_a = [synth.normal(8, i, s, std=0.02).astype(np.float32).astype(np.float64)
           for i, (_, s, _) in enumerate(ADAM)]
    m_a = [np.zeros(s) for _, s, _ in ADAM]
    v_a = [np.zeros(s) for _, s, _ in ADAM]
    t = 0
    W64 = [None] * len(MUON)
    EB = [0.0] * len(MUON)
    EA = [(0.0, 0.0, 0.0)] * len(ADAM)
    for hm, ha in steps_grads:
        ctl = oracle.grad_control(hm + ha, inv, max_norm)
        if ctl.skip:
            continue
        t += 1
        for i, (_, s, views, _) in enumerate(MUON):
            EB[i] = momentum_atol(B_m[i], ctl.mult * hm[i], HP.momentum, EB[i], G_REL)
            Wn, Bn, _, _ = oracle.muon_step_tensor(W_m[i], ctl.mult * hm[i], B_m[i], HP,
                                                   views=views, wd=MUON_WD)
            W64[i] = Wn
            W_m[i] = Wn.astype(np.float32).astype(np.float64)
            B_m[i] = Bn
        for j in range(len(ADAM)):
            EA[j] = adamw_atol(W_a[j], ctl.mult * ha[j], m_a[j], v_a[j], ADAM_HP["lr"],
                               *ADAM_HP["betas"], ADAM_HP["eps"], ADAM_WD, t, EA[j], G_REL)
            Wn, m_a[j], v_a[j] = oracle.adamw_step(W_a[j], ctl.mult * ha[j], m_a[j], v_a[j],
                                                   ADAM_HP["lr"], *ADAM_HP["betas"],
                                                   ADAM_HP["eps"], ADAM_WD, t)
            W_a[j] = Wn.astype(np.float32).astype(np.float64)
    return dict(Wm=W_m, W64=W64, Bm=B_m, Wa=W_a, m=m_a, v=v_a, t=t, EB=EB, EA=EA)


def test_hybrid_steps_under_clipping_and_a_skipped_step():
    """Four steps with the global norm clipped to 0.2 (about 0.4 of its value)
    and an inf in an AdamW gradient at step 2: that step writes nothing, and
    the others match the oracle (AdamW's bias correction counts 3 steps)."""
    import torch
    import muon_adamw_hybrid_gb300 as mh
    inv, max_norm = 1.0 / 64, 0.2
    pm = [torch.tensor(synth.normal(7, i, s, std=0.02), dtype=torch.float32, device="cuda")
          for i, (_, s, _, _) in enumerate(MUON)]
    pa = [torch.tensor(synth.normal(8, i, s, std=0.02), dtype=torch.float32, device="cuda")
          for i, (_, s, _) in enumerate(ADAM)]
    opt = mh.HybridMuonAdamW([dict(param=p, views=v, wd=MUON_WD)
                              for p, (_, _, v, _) in zip(pm, MUON)],
                             [dict(param=p, wd=ADAM_WD) for p in pa], lr=HP.lr,
                             adam_lr=ADAM_HP["lr"], adam_betas=ADAM_HP["betas"],
                             adam_eps=ADAM_HP["eps"], max_grad_norm=max_norm)
    steps = []
    for s in range(4):
        hm, ha = _grads(10 + s, 64.0)
        if s == 2:
            ha[0] = ha[0].copy()
            ha[0][5, 5] = np.inf
        steps.append((hm, ha))
        gm = [_dev(g, d) for g, (*_, d) in zip(hm, MUON)]
        ga = [_dev(g, d) for g, (*_, d) in zip(ha, ADAM)]
        if s == 2:
            before = [t.clone() for t in pm + pa + opt.momentum + opt.exp_avg + opt.exp_avg_sq]
        opt.step(gm, ga, inv_loss_scale=inv)
        torch.cuda.synchronize()
        if s == 2:
            assert int(opt.control.skip.item()) == 1
            after = pm + pa + opt.momentum + opt.exp_avg + opt.exp_avg_sq
            for x, y in zip(before, after):
                assert torch.equal(x, y)
        else:
            assert int(opt.control.skip.item()) == 0
    ref = _oracle_run(steps, max_norm, inv)
    assert opt.applied_steps() == ref["t"] == 3
    for i, (name, s, views, _) in enumerate(MUON):
        check_fp32(to_np(opt.momentum[i]), ref["Bm"][i], ref["EB"][i], f"clipped {name} momentum")
        w0 = synth.normal(7, i, s, std=0.02).astype(np.float32).astype(np.float64)
        tol = max(1e-3, 2e-2 * np.linalg.norm(ref["W64"][i] - w0) / np.linalg.norm(ref["W64"][i]))
        assert rel_fro(to_np(pm[i]), ref["Wm"][i]) < tol, name
    for j, (name, _, _) in enumerate(ADAM):
        check_fp32(to_np(opt.exp_avg[j]), ref["m"][j], ref["EA"][j][0], f"clipped {name} m")
        check_fp32(to_np(opt.exp_avg_sq[j]), ref["v"][j], ref["EA"][j][1], f"clipped {name} v")
        check_fp32(to_np(pa[j]), ref["Wa"][j], ref["EA"][j][2], f"clipped {name} W")


def test_skipped_step_under_normuon_and_muon_plus_changes_nothing():
    """With NorMuon, Muon+ and the cautious-update mask on (so every separate
    pass runs: row statistics in the GEMM, column statistics, both
    finalisations, the apply), a step with an inf gradient leaves parameters,
    momentum, NorMuon state and AdamW moments bit for bit as they were, and
    the steps around it equal those of an optimizer that never saw it."""
    import torch
    import muon_adamw_hybrid_gb300 as mh

    def make():
        pm = [torch.tensor(synth.normal(17, i, s, std=0.02), dtype=torch.float32, device="cuda")
              for i, (_, s, _, _) in enumerate(MUON)]
        pa = [torch.tensor(synth.normal(18, i, s, std=0.02), dtype=torch.float32, device="cuda")
              for i, (_, s, _) in enumerate(ADAM)]
        opt = mh.HybridMuonAdamW([dict(param=p, views=v, wd=MUON_WD)
                                  for p, (_, _, v, _) in zip(pm, MUON)],
                                 [dict(param=p, wd=0.1) for p in pa],
                                 normuon=True, muon_plus=True, cautious=2, max_grad_norm=1.0)
        return pm, pa, opt

    def grads(step, bad=False):
        gm = [torch.tensor(synth.normal(19 + step, i, s, std=1e-3), dtype=torch.float32,
                           device="cuda") for i, (_, s, _, _) in enumerate(MUON)]
        ga = [torch.tensor(synth.normal(29 + step, i, s, std=1e-3), dtype=torch.float32,
                           device="cuda") for i, (_, s, _) in enumerate(ADAM)]
        if bad:
            gm[0].view(-1)[5] = float("inf")
        return gm, ga

    pm, pa, opt = make()
    rm, ra, ref = make()
    opt.step(*grads(0))
    ref.step(*grads(0))
    torch.cuda.synchronize()
    state = [t.clone() for t in pm + pa + opt.momentum + opt.exp_avg + opt.exp_avg_sq
             + [s for s in opt.normuon_sm if s is not None]]
    opt.step(*grads(1, bad=True))
    torch.cuda.synchronize()
    after = pm + pa + opt.momentum + opt.exp_avg + opt.exp_avg_sq + \
        [s for s in opt.normuon_sm if s is not None]
    for a, b in zip(state, after):
        assert torch.equal(a, b)
    assert int(opt.control.skip.item()) == 1 and opt.applied_steps() == 1
    opt.step(*grads(2))
    ref.step(*grads(2))
    torch.cuda.synchronize()
    for a, b in zip(pm + pa + opt.momentum + opt.exp_avg + opt.exp_avg_sq,
                    rm + ra + ref.momentum + ref.exp_avg + ref.exp_avg_sq):
        assert torch.equal(a, b)
    for a, b in zip(opt.normuon_sm, ref.normuon_sm):
        assert a is None or torch.equal(a, b)
