"""Out-of-bounds writes: every buffer a call writes sits inside a larger
allocation whose guard bands before and after it hold a sentinel bit pattern;
after the call (ragged shapes, every variant that adds a pass, tall views,
one-row and one-column views) the guards are bit for bit unchanged, the
read-only gradients are unchanged, and the results are finite. Guard bands of
4096 elements keep the tensors 16-byte aligned (vector paths); 4099 elements
misalign them (the element-wise fallbacks).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

GUARD = 4096   # elements on each side (set per test)
SENT32 = 0x7FC0DEAD
SENT16 = 0x7FAB


@pytest.fixture(params=[4096, 4099], autouse=True)
def guard(request):
    global GUARD
    GUARD = request.param
    yield


def _guarded(values: np.ndarray, dtype):
    """(whole allocation, the tensor inside it) with sentinel guard bands."""
    import torch
    n = values.size
    whole = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        whole.view(torch.int16).fill_(SENT16)
    else:
        whole.view(torch.int32).fill_(SENT32)
    inner = whole[GUARD:GUARD + n].view(values.shape)
    inner.copy_(torch.tensor(values, dtype=torch.float32, device="cuda").to(dtype))
    return whole, inner


def _guards_intact(whole, n) -> bool:
    import torch
    if whole.dtype == torch.bfloat16:
        bits, sent = whole.view(torch.int16), SENT16
    else:
        bits, sent = whole.view(torch.int32), SENT32
    return bool(torch.all(bits[:GUARD] == sent)) and bool(torch.all(bits[GUARD + n:] == sent))


SHAPES = [(1, 130, 136), (2, 300, 200), (3, 33, 65), (1, 1, 64), (1, 64, 1), (1, 700, 300)]


@pytest.mark.parametrize("flags", [dict(), dict(normuon=True, muon_plus=True, cautious=1),
                                   dict(cautious=2)])
@pytest.mark.parametrize("pdt", ["f32", "bf16"])
def test_muon_step_writes_only_its_buffers(flags, pdt):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    tdt = torch.float32 if pdt == "f32" else torch.bfloat16
    keep, ts = [], []
    for t, (v, r, c) in enumerate(SHAPES):
        w = synth.normal(60, t, (v * r, c), std=1.0)
        g = synth.normal(61, t, (v * r, c), std=0.1)
        W = _guarded(w, tdt)
        G = _guarded(g, tdt)
        B = _guarded(np.zeros((v * r, c)), torch.float32)
        S = _guarded(np.zeros(v * r), torch.float32) if flags.get("normuon") else (None, None)
        g0 = G[1].clone()
        keep.append((W, G, B, S, g0, v * r * c, v * r))
        ts.append(mh.muon_tensor(W[1], G[1], B[1], v, S[1], 1.0, 0.01))
    hp = mh.make_hparams(**flags)
    need = mh.muon_workspace_bytes(ts, hp)
    gb = 256 * 64                                # workspace guard bytes, keeps 256-byte alignment
    wsw = torch.full((need + 2 * gb,), 0xA5, dtype=torch.uint8, device="cuda")
    ws_ptr = wsw.data_ptr() + gb
    assert ws_ptr % 256 == 0
    mh.muon_step_batched(ts, hp, ws_ptr, need, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    mh.workspace_status(ws_ptr, torch.cuda.current_stream().cuda_stream)
    assert bool(torch.all(wsw[:gb] == 0xA5)) and bool(torch.all(wsw[gb + need:] == 0xA5))
    for (W, G, B, S, g0, n, rows) in keep:
        assert _guards_intact(W[0], n) and _guards_intact(G[0], n) and _guards_intact(B[0], n)
        if S[0] is not None:
            assert _guards_intact(S[0], rows)
            assert torch.isfinite(S[1]).all()
        assert torch.equal(G[1], g0)
        assert torch.isfinite(W[1].float()).all() and torch.isfinite(B[1]).all()


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_newton_schulz_writes_only_its_output(out_dtype):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    xs, outs = [], []
    for t, (v, r, c) in enumerate(SHAPES):
        x = torch.tensor(synth.normal(62, t, (v * r, c), std=1.0), dtype=torch.float32,
                         device="cuda")
        xs.append(x)
        outs.append(_guarded(np.zeros((v * r, c)), tdt))
    mh.newton_schulz(xs, [o[1] for o in outs], views=[s[0] for s in SHAPES])
    torch.cuda.synchronize()
    for o, (v, r, c) in zip(outs, SHAPES):
        assert _guards_intact(o[0], v * r * c)
        assert torch.isfinite(o[1].float()).all()


@pytest.mark.parametrize("pdt", ["f32", "bf16"])
def test_adamw_writes_only_its_buffers(pdt):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    tdt = torch.float32 if pdt == "f32" else torch.bfloat16
    keep, ts = [], []
    for t, n in enumerate([1, 7, 10007, 65536 + 3]):
        W = _guarded(synth.normal(63, t, (n,), std=0.02), tdt)
        G = _guarded(synth.normal(64, t, (n,), std=1e-3), tdt)
        M = _guarded(np.zeros(n), torch.float32)
        V = _guarded(np.zeros(n), torch.float32)
        keep.append((W, G, M, V, n))
        ts.append(mh.adamw_tensor(W[1], G[1], M[1], V[1], 1.0, 0.1))
    mh.adamw_step(ts, 3e-4, 0.9, 0.95, 1e-8, 1, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for (W, G, M, V, n) in keep:
        for buf in (W, G, M, V):
            assert _guards_intact(buf[0], n)
        assert torch.isfinite(W[1].float()).all()
