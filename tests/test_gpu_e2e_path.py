"""The end-to-end path that bench.py times computes the same step as the
device-resident path: gradients read in place from page-locked host memory,
each Muon step split into its gradient phase and the rest, the previous
step's parameters copied out on a second stream between the two, and the
update fenced on that copy. On the 124M set with gradient clipping on, three
steps of both paths give bit-identical parameters, momentum and moments, and
every copy-out equals the parameters of the step it follows.
"""
import pytest

import bench
from synth import workloads as W

pytestmark = pytest.mark.gpu


def test_split_fenced_host_path_equals_device_path():
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
    gin = bench.PinnedMirror(run.mG + run.aG)
    gin.fill_from_device()
    pout = bench.PinnedMirror(run.mW + run.aW)
    torch.cuda.synchronize()
    nm = len(run.mG)
    run.use_host_grads(gin.host[:nm], gin.host[nm:])
    copy_stream = torch.cuda.Stream()
    snapshots = []

    def copy_out():
        ready = torch.cuda.Event()
        ready.record(stream)
        copy_stream.wait_event(ready)
        with torch.cuda.stream(copy_stream):
            pout.d2h()
            landed = torch.cuda.Event()
            landed.record(copy_stream)
        return landed

    expect = []
    for k in range(3):
        ref.step(stream)
        expect.append([t.clone() for t in ref.mW + ref.aW])
        fence = {}

        def between(k=k):
            if k == 0:
                return None
            fence["e"] = copy_out()
            return fence["e"]
        run.step(stream, host_grads=True, between=between)
        if k > 0:
            fence["e"].synchronize()
            snapshots.append([h.clone() for h in pout.host])
    stream.wait_event(copy_out())
    torch.cuda.synchronize()
    snapshots.append([h.clone() for h in pout.host])
    ref.check_status(stream)
    run.check_status(stream)

    for a, b in zip(ref.mW + ref.mB + ref.aW + ref.am + ref.av,
                    run.mW + run.mB + run.aW + run.am + run.av):
        assert torch.equal(a, b)
    assert int(run.control.step.item()) == int(ref.control.step.item()) == 3
    for k, snap in enumerate(snapshots):
        for want, got in zip(expect[k], snap):
            assert torch.equal(want.cpu(), got)
    run.ts_host = run.at_host = None
    gin.close()
    pout.close()
