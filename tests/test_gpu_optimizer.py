"""The torch-facing optimizer facade and checkpoint continuation."""
import pytest

import synth

pytestmark = pytest.mark.gpu


def _params():
    import torch
    torch.manual_seed(0)
    p = {
        "q": torch.tensor(synth.normal(5, 1, (256, 256), std=0.02), device="cuda"),
        "gate_up": torch.tensor(synth.normal(5, 2, (2 * 384, 128), std=0.02), device="cuda"),
        "embed": torch.tensor(synth.normal(5, 3, (1000, 64), std=0.02), device="cuda"),
        "norm": torch.ones(64, device="cuda"),
    }
    return p


def _grads(step):
    import torch
    return {k: torch.tensor(synth.normal(6, 100 * step + i, shape, std=1e-3), device="cuda")
            for i, (k, shape) in enumerate([("q", (256, 256)), ("gate_up", (768, 128)),
                                            ("embed", (1000, 64)), ("norm", (64,))])}


def _opt(p, **kw):
    import muon_adamw_hybrid_gb300 as mh
    return mh.HybridMuonAdamW([dict(param=p["q"], wd=0.01), dict(param=p["gate_up"], views=2, wd=0.01)],
                              [dict(param=p["embed"], wd=0.1), dict(param=p["norm"], wd=0.1)], **kw)


def _step(opt, step):
    g = _grads(step)
    opt.step([g["q"], g["gate_up"]], [g["embed"], g["norm"]])


def test_state_dict_continuation_is_bitwise():
    import torch
    pa, pb = _params(), _params()
    a = _opt(pa, normuon=True)
    for s in range(2):
        _step(a, s)
    b = _opt(pb, normuon=True)
    for s in range(2):
        _step(b, s)
    sd = b.state_dict()
    snap = {k: v.clone() for k, v in pb.items()}
    c = _opt(snap, normuon=True)
    c.load_state_dict(sd)
    _step(a, 2)
    _step(c, 2)
    torch.cuda.synchronize()
    for k in pa:
        assert torch.equal(pa[k], snap[k]), k


def test_routing_helper_and_facade_step():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    p = {k: v.requires_grad_(True) for k, v in _params().items()}
    muon, adamw = mh.route_parameters(
        [("layers.0.attn.q_proj.weight", p["q"]), ("layers.0.mlp.gate_up", p["gate_up"]),
         ("embed_tokens.weight", p["embed"]), ("layers.0.norm.weight", p["norm"])],
        views={"layers.0.mlp.gate_up": 2})
    assert [n for n, _, _ in muon] == ["layers.0.attn.q_proj.weight", "layers.0.mlp.gate_up"]
    assert [n for n, _ in adamw] == ["embed_tokens.weight", "layers.0.norm.weight"]
    opt = mh.HybridMuonAdamW([dict(param=t, views=v) for _, t, v in muon],
                             [dict(param=t) for _, t in adamw])
    before = {k: v.clone() for k, v in p.items()}
    _step(opt, 0)
    torch.cuda.synchronize()
    for k in p:
        assert not torch.equal(before[k], p[k]), k


def test_pinned_host_gradients_are_read_in_place():
    """Gradients in page-locked host memory that the device maps at the same
    address are read by the kernels directly; the result equals the step on
    device-resident gradients bit for bit."""
    import torch
    import muon_adamw_hybrid_gb300 as mh
    probe = torch.empty(16, pin_memory=True)
    if not mh.pointer_device_accessible(probe.data_ptr()):
        pytest.skip("this system does not map page-locked host memory into the device")
    pa, pb = _params(), _params()
    a, b = _opt(pa), _opt(pb)
    for s in range(2):
        g = _grads(s)
        host = {k: v.cpu().pin_memory() for k, v in g.items()}
        a.step([g["q"], g["gate_up"]], [g["embed"], g["norm"]])
        b.step([host["q"], host["gate_up"]], [host["embed"], host["norm"]])
    torch.cuda.synchronize()
    for k in pa:
        assert torch.equal(pa[k], pb[k]), k
