"""bf16 optimizer state with stochastic rounding on the GPU, against the
oracle (dew.training.optim, "stochastic_round_bf16" and "bf16_moments").

The rounding decision depends on the fp32 value before rounding. The GPU
computes that value in fp32, the oracle in fp64 (then rounded to fp32), so the
two can differ by a few fp32 ulps. Where such a difference cannot move the
decision (the dropped 16 bits plus the noise are at least D units away from a
carry), the GPU's bf16 state must equal the oracle's bit for bit; that is all
but about 2D/65536 of the elements, and a wrong hash, key, stream or index
would break about a third of them. The rest must be one of the two bf16
neighbours. For the parameter after a Newton-Schulz update the pre-rounding
difference is the NS error itself, so there the check is the final-parameter
bar plus the agreement rate of the decisions.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import rel_fro, to_np

pytestmark = pytest.mark.gpu

D_ULPS = 16
REL_TERMS = 1e-6   # fp32 arithmetic and fp32 constants (e.g. 1 - 0.9f), relative to the terms


def _bits_bf16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().astype(np.uint16).astype(np.uint32)


def _expected_bits(x64, seed, stream, terms=None, index0=0):
    """bf16 bits the oracle's stochastic rounding gives, and a mask of the
    elements whose decision the GPU's fp32 arithmetic could flip: those whose
    dropped bits plus noise lie within `margin` fp32 ulps of a carry, with
    margin = max(D_ULPS, REL_TERMS * terms / ulp), `terms` the sum of the
    magnitudes of the terms that make up the value (a sum that nearly
    cancels carries the error of its terms)."""
    x32 = np.ascontiguousarray(np.asarray(x64, dtype=np.float64).ravel().astype(np.float32))
    noise = oracle.sr_noise16(oracle.sr_key(seed, stream),
                              np.arange(index0, index0 + x32.size, dtype=np.uint64))
    out = oracle.round_bf16_with_noise(x32, noise)
    bits = out.astype(np.float32).view(np.uint32) >> np.uint32(16)
    margin = np.full(x32.size, float(D_ULPS))
    if terms is not None:
        ulp = np.spacing(np.abs(x32)).astype(np.float64)
        margin = np.maximum(margin, np.ceil(REL_TERMS * np.asarray(terms).ravel() / ulp))
    frac = ((x32.view(np.uint32).astype(np.int64) & 0xFFFF) + noise.astype(np.int64)) & 0xFFFF
    ambiguous = (frac < margin) | (frac >= 65536 - margin)
    return bits.astype(np.uint32), ambiguous


def _check_state(got_t, x64, seed, stream, what, terms=None, index0=0):
    got = _bits_bf16(got_t).ravel()
    want, amb = _expected_bits(x64, seed, stream, terms, index0)
    clear = ~amb
    mism = np.flatnonzero(got[clear] != want[clear])
    assert mism.size == 0, (what, mism.size, int(clear.sum()))
    # ambiguous elements: within one bf16 spacing of the oracle's value, after
    # the arithmetic error allowed for the terms
    x = np.asarray(x64, dtype=np.float64).ravel()[amb]
    gv = (got[amb] << np.uint32(16)).astype(np.uint32).view(np.float32).astype(np.float64)
    err = 0.0 if terms is None else REL_TERMS * np.asarray(terms).ravel()[amb]
    mag = np.maximum(np.maximum(np.abs(x), np.abs(gv)), 1e-38)
    spacing = 2.0 ** (np.floor(np.log2(mag)) - 7)
    assert np.all(np.abs(gv - x) <= err + spacing), what
    assert amb.mean() < 0.01, (what, amb.mean())


ADAM_SPECS = [("a", 4099, "bf16", False), ("b", 65536 + 3, "f32", False),
              ("c", 1000, "bf16", True)]    # True: base address off by one element


def _adam_inputs(seed):
    out = []
    for t, (_, n, gdt, _) in enumerate(ADAM_SPECS):
        w = synth.normal(60 + seed, t, (n,), std=0.02, dtype="bf16").astype(np.float64)
        g = synth.normal(61 + seed, t, (n,), std=1e-3, dtype=gdt).astype(np.float64)
        m = synth.normal(62 + seed, t, (n,), std=1e-4, dtype="bf16").astype(np.float64)
        v = np.abs(synth.normal(63 + seed, t, (n,), std=1e-6, dtype="bf16").astype(np.float64))
        out.append((w, g, m, v))
    return out


def _dev(x, dtype, misaligned=False):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = torch.tensor(np.asarray(x), dtype=torch.float64, device="cuda").to(tdt)
    if not misaligned:
        return t
    buf = torch.zeros(t.numel() + 1, dtype=tdt, device="cuda")
    buf[1:] = t
    return buf[1:]


def _run_adam(inputs, step, ctl=None):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    devs, structs = [], []
    for (w, g, m, v), (_, _, gdt, mis) in zip(inputs, ADAM_SPECS):
        dw, dg = _dev(w, "bf16", mis), _dev(g, gdt, mis)
        dm, dv = _dev(m, "bf16", mis), _dev(v, "bf16", mis)
        devs.append((dw, dg, dm, dv))
        structs.append(mh.adamw_tensor(dw, dg, dm, dv, 1.0, 0.1, param_sr=True))
    s = torch.cuda.current_stream().cuda_stream
    if ctl is None:
        mh.adamw_step(structs, 3e-4, 0.9, 0.95, 1e-8, step, s)
    else:
        mh.grad_prepare([d[1] for d in devs], ctl, 1.0, 0.0)
        mh.adamw_step_ctl(structs, 3e-4, 0.9, 0.95, 1e-8, ctl.struct(), s)
    torch.cuda.synchronize()
    return devs


@pytest.mark.parametrize("step", [1, 7])
def test_adamw_bf16_moments_and_param_sr_match_the_oracle(step):
    inputs = _adam_inputs(step)
    devs = _run_adam(inputs, step)
    for t, ((w, g, m, v), (dw, _, dm, dv)) in enumerate(zip(inputs, devs)):
        W, M, V = oracle.adamw_step(w, g, m, v, 3e-4, 0.9, 0.95, 1e-8, 0.1, step)
        upd = np.abs(W - w * (1 - 3e-4 * 0.1))
        _check_state(dm, M, step, oracle.sr_stream(t, oracle.MOMENT_FIRST), f"m{t}",
                     terms=np.abs(0.9 * m) + np.abs(0.1 * g))
        _check_state(dv, V, step, oracle.sr_stream(t, oracle.MOMENT_SECOND), f"v{t}",
                     terms=np.abs(0.95 * v) + np.abs(0.05 * g * g))
        _check_state(dw, W, step, oracle.sr_stream(t, oracle.MOMENT_PARAM), f"W{t}",
                     terms=np.abs(w) + 10.0 * upd)


def test_device_step_count_seeds_like_the_host_count():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    inputs = _adam_inputs(3)
    host = _run_adam(inputs, 5)
    ctl = mh.GradientControl("cuda", step=4)      # prepare advances it to 5
    dev = _run_adam(inputs, None, ctl)
    for a, b in zip(host, dev):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def _muon_run(specs, hp_kw, seed, momentum_dtype, param_sr):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    hp = mh.make_hparams(**hp_kw)
    hp.sr_seed = seed
    tens, keep = [], []
    for t, (name, views, r, c, pdt) in enumerate(specs):
        n = views * r * c
        # unit-scale weights: the update is below a bf16 spacing, where the
        # rounding decides, and the NS error is far below one spacing
        w = synth.normal(70, t, (views * r, c), std=1.0, dtype=pdt).astype(np.float64)
        g = synth.normal(71, t, (views * r, c), std=1e-3, dtype="bf16").astype(np.float64)
        b = synth.normal(72, t, (views * r, c), std=1e-3, dtype="bf16").astype(np.float64)
        dw, dg = _dev(w, pdt), _dev(g, "bf16")
        db = _dev(b, momentum_dtype)
        sm = torch.zeros(views * r, dtype=torch.float32, device="cuda") if hp_kw.get("normuon") \
            else None
        # every buffer the call reads stays referenced until it has run (the C
        # ABI holds raw pointers)
        keep.append((w, g, b, dw, dg, db, sm, n))
        tens.append(mh.muon_tensor(dw, dg, db, views, sm, 1.0, 0.01, param_sr=param_sr))
    need = mh.muon_workspace_bytes(tens, hp)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    mh.muon_step_batched(tens, hp, ws.data_ptr(), ws.numel(),
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return keep


MUON_SPECS = [("sq", 1, 256, 256, "bf16"), ("tall", 2, 384, 128, "bf16"),
              ("wide", 1, 96, 200, "bf16"), ("odd", 1, 33, 20, "bf16")]


@pytest.mark.parametrize("hp_kw", [dict(), dict(normuon=True)])
def test_muon_bf16_momentum_and_param_sr(hp_kw):
    seed = 12345
    keep = _muon_run(MUON_SPECS, hp_kw, seed, "bf16", True)
    ohp = oracle.MuonHparams(normuon=hp_kw.get("normuon", False))
    agree_total = n_total = 0
    for t, (spec, kept) in enumerate(zip(MUON_SPECS, keep)):
        (name, views, r, c, pdt), (w, g, b, dw, _, db, sm, n) = spec, kept
        W64, B64, _, _ = oracle.muon_step_tensor(w, g, b, ohp, views=views, wd=0.01,
                                                 sm=None if sm is None else np.zeros(views * r))
        _check_state(db, B64, seed, oracle.sr_stream(t, oracle.MOMENT_FIRST), f"B {name}",
                     terms=np.abs(0.95 * b) + np.abs(0.05 * g))
        # parameter: the final-parameter bar, and the rounding decisions
        got = to_np(dw).reshape(W64.shape)
        tol = max(1e-3, 2e-2 * np.linalg.norm(W64 - 0.9998 * w) / np.linalg.norm(W64),
                  2.0 * rel_fro(oracle.round_bf16(W64), W64))
        assert rel_fro(got, W64) < tol, (name, rel_fro(got, W64), tol)
        want, _ = _expected_bits(W64, seed, oracle.sr_stream(t, oracle.MOMENT_PARAM))
        gb = _bits_bf16(dw).ravel()
        agree_total += int(np.sum(gb == want))
        n_total += n
    # a wrong key, stream or index agrees on about two thirds of the decisions
    assert agree_total / n_total > 0.97, agree_total / n_total


def test_bf16_momentum_without_param_sr_keeps_nearest_even_params():
    keep_sr = _muon_run(MUON_SPECS[:1], {}, 7, "bf16", False)
    keep_f32 = _muon_run(MUON_SPECS[:1], {}, 7, "f32", False)
    import torch
    # same fp32 Q either way (the update reads the unrounded momentum), so the
    # nearest-even parameters are identical
    assert torch.equal(keep_sr[0][3], keep_f32[0][3])
