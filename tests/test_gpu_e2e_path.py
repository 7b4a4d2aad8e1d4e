"""The end-to-end path that bench.py times (bench.HostPipeline) computes the
same step as the device-resident path: Muon gradients read in place from
page-locked host memory, each Muon step split into its gradient phase and the
rest, the AdamW gradients copied in and the previous step's parameters copied
out on side streams between the two, and the update fenced on the copy-out.
On the 124M set with gradient clipping on, three steps of both paths give
bit-identical parameters, momentum and moments, and every copy-out equals the
parameters of the step it follows.
"""
import pytest

import bench
from synth import workloads as W

pytestmark = pytest.mark.gpu


def test_host_pipeline_equals_device_path():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    probe = torch.empty(16, pin_memory=True)
    if not mh.pointer_device_accessible(probe.data_ptr()):
        pytest.skip("this system does not map page-locked host memory into the device")
    wl = W.gpt124m()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    ref = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    run = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    pipe = bench.HostPipeline(run)
    assert pipe.in_place
    run.aG[0].zero_()           # AdamW must read the copied-in host values, not stale ones

    expect, snapshots = [], []
    for k in range(3):
        ref.step(stream)
        expect.append([t.clone() for t in ref.mW + ref.aW])
        pipe.step(stream)
        if k > 0:               # this step copied out the previous step's parameters
            pipe.last_copy.synchronize()
            snapshots.append([h.clone() for h in pipe.pout.host])
    pipe.finish(stream).synchronize()
    snapshots.append([h.clone() for h in pipe.pout.host])
    torch.cuda.synchronize()
    ref.check_status(stream)
    run.check_status(stream)

    for a, b in zip(ref.mW + ref.mB + ref.aW + ref.am + ref.av,
                    run.mW + run.mB + run.aW + run.am + run.av):
        assert torch.equal(a, b)
    assert int(run.control.step.item()) == int(ref.control.step.item()) == 3
    for want_step, snap in zip(expect, snapshots):
        for want, got in zip(want_step, snap):
            assert torch.equal(want.cpu(), got)
    pipe.close()


def test_grouped_host_pipeline_equals_device_path():
    """Same check for the grouped step (bench.HostPipeline.step_grouped): half
    of the Muon tensors read their gradients in place, the rest and AdamW's are
    copied in while the first half's Newton-Schulz stages run, and each
    group's update is fenced on the copy-out of its own parameters."""
    import torch
    import muon_adamw_hybrid_gb300 as mh
    probe = torch.empty(16, pin_memory=True)
    if not mh.pointer_device_accessible(probe.data_ptr()):
        pytest.skip("this system does not map page-locked host memory into the device")
    wl = W.gpt124m()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    ref = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    run = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    pipe = bench.HostPipeline(run)
    n = len(wl.muon)
    groups = ([i for i in range(n) if i % 3 == 0], [i for i in range(n) if i % 3 != 0])
    for i in groups[1]:
        run.mG[i].zero_()       # group B must read the copied-in host values
    run.aG[0].zero_()

    expect, snapshots = [], []
    for k in range(3):
        ref.step(stream)
        expect.append([t.clone() for t in ref.mW + ref.aW])
        pipe.step_grouped(stream, groups)
        if k > 0:
            pipe.last_copy.synchronize()
            snapshots.append([h.clone() for h in pipe.pout.host])
    pipe.finish(stream).synchronize()
    snapshots.append([h.clone() for h in pipe.pout.host])
    torch.cuda.synchronize()
    ref.check_status(stream)
    run.check_status(stream)
    for a, b in zip(ref.mW + ref.mB + ref.aW + ref.am + ref.av,
                    run.mW + run.mB + run.aW + run.am + run.av):
        assert torch.equal(a, b)
    for want_step, snap in zip(expect, snapshots):
        for want, got in zip(want_step, snap):
            assert torch.equal(want.cpu(), got)
    pipe.close()
