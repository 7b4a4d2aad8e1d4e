"""The parameter-write fence of the Muon step (mh_muon_hparams.param_fence).

Another stream spins for about 20 ms, then snapshots the parameter and the
momentum and records the fence; the step on the main stream is enqueued right
after. The snapshot must hold the parameter from before the step (the step's
first parameter write waited for the fence) but the momentum from after it
(the prologue did not wait), and the finished step must equal the same step
taken without a fence, bit for bit.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 40_000_000      # about 20 ms at 2 GHz


def _tensors(dtype):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    out = []
    for t, (views, r, c) in enumerate([(2, 256, 512), (1, 768, 256)]):
        w = torch.tensor(synth.normal(90, t, (views * r, c), std=0.02), dtype=dtype, device="cuda")
        g = torch.tensor(synth.normal(91, t, (views * r, c), std=1e-3), dtype=dtype, device="cuda")
        b = torch.zeros((views * r, c), dtype=torch.float32, device="cuda")
        sm = torch.zeros(views * r, dtype=torch.float32, device="cuda")
        out.append(dict(w=w, g=g, b=b, sm=sm, views=views))
    return out


def _step(hp, tens, stream):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    ts = [mh.muon_tensor(d["w"], d["g"], d["b"], d["views"], d["sm"], 1.0, 0.01) for d in tens]
    ws = torch.empty(mh.muon_workspace_bytes(ts, hp), dtype=torch.uint8, device="cuda")
    mh.muon_step_batched(ts, hp, ws.data_ptr(), ws.numel(), stream.cuda_stream)
    return ws


@pytest.mark.parametrize("normuon", [False, True])
def test_fence_holds_back_only_the_parameter_write(normuon):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()

    # the same step without a fence
    ref = _tensors(torch.bfloat16)
    hp = mh.make_hparams(normuon=normuon)
    _step(hp, ref, main)
    torch.cuda.synchronize()

    tens = _tensors(torch.bfloat16)
    w0 = [d["w"].clone() for d in tens]
    snap_w = [torch.empty_like(d["w"]) for d in tens]
    snap_b = [torch.empty_like(d["b"]) for d in tens]
    fence = torch.cuda.Event()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(SPIN_CYCLES)
        for d, sw, sb in zip(tens, snap_w, snap_b):
            sw.copy_(d["w"])
            sb.copy_(d["b"])
        fence.record(side)
    hp = mh.make_hparams(normuon=normuon)
    hp.param_fence = fence.cuda_event
    ws = _step(hp, tens, main)
    torch.cuda.synchronize()
    mh.workspace_status(ws.data_ptr(), main.cuda_stream)

    for d, r, sw, sb, w in zip(tens, ref, snap_w, snap_b, w0):
        assert torch.equal(sw, w)                     # no parameter write before the fence
        assert torch.equal(sb, r["b"])                # the prologue ran alongside the spin
        assert torch.equal(d["w"], r["w"]) and torch.equal(d["b"], r["b"])
        assert not torch.equal(d["w"], w)
        if normuon:
            assert torch.equal(d["sm"], r["sm"])


def test_optimizer_step_takes_a_fence():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    side = torch.cuda.Stream()
    params = [torch.nn.Parameter(torch.tensor(synth.normal(92, 0, (256, 512), std=0.02),
                                              dtype=torch.bfloat16, device="cuda")),
              torch.nn.Parameter(torch.tensor(synth.normal(92, 1, (4096,), std=0.02),
                                              dtype=torch.bfloat16, device="cuda"))]
    for k, p in enumerate(params):
        p.grad = torch.tensor(synth.normal(93, k, tuple(p.shape), std=1e-3),
                              dtype=torch.bfloat16, device="cuda")
    opt = mh.HybridMuonAdamW([dict(param=params[0])], [dict(param=params[1])])
    before = [p.detach().clone() for p in params]
    snap = [torch.empty_like(p) for p in params]
    fence = torch.cuda.Event()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(SPIN_CYCLES)
        for s, p in zip(snap, params):
            s.copy_(p.detach())
        fence.record(side)
    opt.step(param_fence=fence)
    torch.cuda.synchronize()
    for s, b, p in zip(snap, before, params):
        assert torch.equal(s, b)
        assert not torch.equal(p.detach(), b)
    assert opt.hp.param_fence is None
    np.testing.assert_equal(opt.applied_steps(), 1)


@pytest.mark.parametrize("variant", [dict(), dict(normuon=True), dict(cautious=2)])
def test_two_phase_step_equals_one_call(variant):
    """MH_STEP_GRADIENTS then MH_STEP_FINISH gives the one-call step bit for
    bit; a snapshot taken between the two (behind a spin on another stream,
    ordered after the gradient phase by an event) sees the new momentum and
    the old parameters, and the finish phase's fence holds its parameter
    write back until the snapshot is done."""
    import torch
    import muon_adamw_hybrid_gb300 as mh
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ref = _tensors(torch.bfloat16)
    _step(mh.make_hparams(**variant), ref, main)
    torch.cuda.synchronize()

    tens = _tensors(torch.bfloat16)
    w0 = [d["w"].clone() for d in tens]
    ts = [mh.muon_tensor(d["w"], d["g"], d["b"], d["views"], d["sm"], 1.0, 0.01) for d in tens]
    hp = mh.make_hparams(**variant)
    ws = torch.empty(mh.muon_workspace_bytes(ts, hp), dtype=torch.uint8, device="cuda")
    snap_w = [torch.empty_like(d["w"]) for d in tens]
    snap_b = [torch.empty_like(d["b"]) for d in tens]
    torch.cuda.synchronize()
    hp.phase = mh.MH_STEP_GRADIENTS
    mh.muon_step_batched(ts, hp, ws.data_ptr(), ws.numel(), main.cuda_stream)
    grads_read = torch.cuda.Event()
    grads_read.record(main)
    fence = torch.cuda.Event()
    with torch.cuda.stream(side):
        side.wait_event(grads_read)
        torch.cuda._sleep(SPIN_CYCLES)
        for d, sw, sb in zip(tens, snap_w, snap_b):
            sw.copy_(d["w"])
            sb.copy_(d["b"])
        fence.record(side)
    hp.phase = mh.MH_STEP_FINISH
    hp.param_fence = fence.cuda_event
    mh.muon_step_batched(ts, hp, ws.data_ptr(), ws.numel(), main.cuda_stream)
    torch.cuda.synchronize()
    mh.workspace_status(ws.data_ptr(), main.cuda_stream)
    for d, r, sw, sb, w in zip(tens, ref, snap_w, snap_b, w0):
        assert torch.equal(sw, w)
        assert torch.equal(sb, r["b"])
        assert torch.equal(d["w"], r["w"]) and torch.equal(d["b"], r["b"])
        assert torch.equal(d["sm"], r["sm"])
