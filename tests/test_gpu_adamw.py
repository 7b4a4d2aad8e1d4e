"""AdamW kernel vs the fp64 oracle.

Bars (tests.parity): the moments and fp32 parameters element by element,
|got - want| <= 1e-6 |want| + 2 atol with atol the running bound on the
kernel's fp32 rounding; bf16 parameters at most one bf16 spacing from the
oracle's rounded value, on at most 0.1 % of the elements.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import check_adam_result, to_np
from tests.parity import adamw_atol

pytestmark = pytest.mark.gpu


def _run(sizes, pdt, gdt, steps=3, offsets=None, lr=1e-3, wd=0.1, b1=0.9, b2=0.95, eps=1e-8):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    offsets = offsets or [0] * len(sizes)
    W0 = [synth.normal(1, i, (n,), std=0.02, dtype=pdt) for i, n in enumerate(sizes)]
    # Storage with a leading offset exercises unaligned (scalar) paths.
    stores = [torch.zeros(o + n, dtype=tdt[pdt], device="cuda") for n, o in zip(sizes, offsets)]
    Ws = [s[o:] for s, o in zip(stores, offsets)]
    for w, w0 in zip(Ws, W0):
        w.copy_(torch.tensor(w0, dtype=torch.float32))
    ms = [torch.zeros(n, device="cuda") for n in sizes]
    vs = [torch.zeros(n, device="cuda") for n in sizes]
    Gs = [torch.empty(n, dtype=tdt[gdt], device="cuda") for n in sizes]
    ref = [(w0.astype(np.float64), np.zeros(n), np.zeros(n)) for w0, n in zip(W0, sizes)]
    bounds = [(0.0, 0.0, 0.0)] * len(sizes)
    for t in range(1, steps + 1):
        G = [synth.normal(2, 1000 * t + i, (n,), std=1e-3, dtype=gdt) for i, n in enumerate(sizes)]
        for g, gh in zip(Gs, G):
            g.copy_(torch.tensor(gh, dtype=torch.float32))
        ts = [mh.adamw_tensor(w, g, m, v, 1.0, wd) for w, g, m, v in zip(Ws, Gs, ms, vs)]
        if t == steps:   # the device's state before the last step
            last = [(to_np(w), to_np(m), to_np(v), gh.astype(np.float64))
                    for w, m, v, gh in zip(Ws, ms, vs, G)]
        mh.adamw_step(ts, lr, b1, b2, eps, t, torch.cuda.current_stream().cuda_stream)
        new, nb = [], []
        for (w, m, v), g, e in zip(ref, G, bounds):
            nb.append(adamw_atol(w, g, m, v, lr, b1, b2, eps, wd, t, e))
            w, m, v = oracle.adamw_step(w, g, m, v, lr, b1, b2, eps, wd, t)
            w = oracle.round_bf16(w) if pdt == "bf16" else w.astype(np.float32).astype(np.float64)
            new.append((w, m, v))
        ref, bounds = new, nb
    torch.cuda.synchronize()
    for k, ((w, m, v), e) in enumerate(zip(ref, bounds)):
        got = (to_np(Ws[k]), to_np(ms[k]), to_np(vs[k]))
        # the whole run from the initial state ...
        r = dict(W=w, m=m, v=v, m_atol=e[0], v_atol=e[1], W_atol=e[2])
        check_adam_result(*got, r, pdt, f"adamw {pdt}/{gdt} tensor {k} of {len(sizes)}",
                          steps=steps)
        # ... and the last step from the device's own state before it
        w0, m0, v0, g = last[k]
        e1 = adamw_atol(w0, g, m0, v0, lr, b1, b2, eps, wd, steps)
        w1, m1, v1 = oracle.adamw_step(w0, g, m0, v0, lr, b1, b2, eps, wd, steps)
        w1 = oracle.round_bf16(w1) if pdt == "bf16" else w1.astype(np.float32).astype(np.float64)
        check_adam_result(*got, dict(W=w1, m=m1, v=v1, m_atol=e1[0], v_atol=e1[1], W_atol=e1[2]),
                          pdt, f"adamw {pdt}/{gdt} tensor {k} of {len(sizes)}, last step")
        if offsets[k]:
            assert torch.all(stores[k][:offsets[k]] == 0)


@pytest.mark.parametrize("pdt,gdt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_adamw_parity_ragged_sizes(pdt, gdt):
    _run([1, 7, 8, 4095, 16384, 16385, 100003], pdt, gdt)


def test_adamw_unaligned_and_empty():
    _run([0, 33, 1000, 5], "f32", "f32", offsets=[0, 1, 3, 2])
    _run([129, 64], "bf16", "bf16", offsets=[1, 5])


def test_adamw_many_tensors_split_launches():
    sizes = [17 + (i * 37) % 300 for i in range(400)]
    _run(sizes, "bf16", "bf16", steps=2)


def test_adamw_large_step_count_bias_correction():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    n = 4096
    w = torch.tensor(synth.normal(3, 1, (n,)), device="cuda")
    g = torch.tensor(synth.normal(3, 2, (n,), std=1e-3), device="cuda")
    m = torch.tensor(synth.normal(3, 3, (n,), std=1e-3), device="cuda")
    v = torch.tensor(np.abs(synth.normal(3, 4, (n,), std=1e-6)), device="cuda")
    w0, g0, m0, v0 = to_np(w), to_np(g), to_np(m), to_np(v)
    ref = oracle.adamw_step(w0, g0, m0, v0, 3e-4, 0.9, 0.95, 1e-8, 0.1, 1000)
    e = adamw_atol(w0, g0, m0, v0, 3e-4, 0.9, 0.95, 1e-8, 0.1, 1000)
    mh.adamw_step([mh.adamw_tensor(w, g, m, v, 1.0, 0.1)], 3e-4, 0.9, 0.95, 1e-8, 1000,
                  torch.cuda.current_stream().cuda_stream)
    r = dict(W=ref[0].astype(np.float32).astype(np.float64), m=ref[1], v=ref[2], m_atol=e[0],
             v_atol=e[1], W_atol=e[2])
    check_adam_result(to_np(w), to_np(m), to_np(v), r, "f32", "adamw step 1000")
