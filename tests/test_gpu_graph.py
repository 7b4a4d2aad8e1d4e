"""The whole hybrid step can be captured in a CUDA graph and replayed.

With gradient control on, AdamW takes its step count from the device
(mh_adamw_step_ctl), so nothing that changes from step to step is baked into
the graph. Three replays of a captured step on the 124M set give bit for bit
the parameters and state of three eager steps. This also holds with the Muon
step in its two phases and a parameter fence recorded inside the capture, and
with NorMuon, Muon+ and the cautious-update mask on (the streaming apply and
column-statistics launches, whose tensor maps are encoded at capture time).
"""
import pytest

import bench
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _state(dw):
    return dw.mW + dw.mB + dw.aW + dw.am + dw.av + [s for s in dw.sm if s is not None]


@pytest.mark.parametrize("split,variants", [(False, {}), (True, {}),
                                            (False, dict(normuon=True, muon_plus=True,
                                                         cautious=2))])
def test_graph_replay_equals_eager_steps(split, variants):
    import torch
    wl = W.gpt124m()
    wl.muon_hp = dict(wl.muon_hp, **variants)
    dev = torch.device("cuda", 0)
    eager = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    graphed = bench.DeviceWorkload(wl, dev, max_grad_norm=1.0)
    stream = torch.cuda.current_stream()
    for _ in range(4):
        eager.step(stream)
    # one eager step first: the library's one-time setup (function attributes,
    # occupancy queries) happens outside the capture
    graphed.step(stream)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            if split:
                fence = torch.cuda.Event()

                def between():
                    fence.record(cap)       # recorded inside the capture
                    return fence
                graphed.step(cap, between=between)
            else:
                graphed.step(cap)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    eager.check_status(stream)
    graphed.check_status(stream)
    assert int(graphed.control.step.item()) == int(eager.control.step.item()) == 4
    for a, b in zip(_state(eager), _state(graphed)):
        assert torch.equal(a, b)
