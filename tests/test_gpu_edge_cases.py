"""Degenerate step configurations against the oracle.

* ns_steps = 0: U is the normalised momentum itself (no GEMM; every pass
  reading U scales it by 1/(||Q|| + eps), the statistics passes of NorMuon and
  Muon+ included); with NorMuon the separate row-statistics pass runs instead
  of the GEMM epilogue's row sums.
* ns_steps = 1: the first iteration's normalisation and the last apply stage
  are the same launch (fused update, or row sums under NorMuon).
* The cautious-update mask under NorMuon / Muon+ (the apply pass's own
  instantiation, which reads the gradient: staged as a TMA box when it is
  bf16 with whole 16-byte rows, read directly otherwise).
* bf16 and fp32 parameters in one NorMuon / Muon+ apply launch: the streaming
  pass's fp32 stage layout holding bf16 tiles, and a bf16 parameter whose
  rows are not whole 16-byte groups (read directly instead of staged).
* Seventy tensors: several elementwise batches, and several parts of a
  streaming cautious-update launch.
* A call mixing empty tensors (zero rows, zero views' worth of elements) with
  ordinary ones: the empty ones are skipped, the rest match the oracle.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.helpers import DeviceRun
from tests.test_gpu_muon import _check, _run_and_check_last_step, _wl

pytestmark = pytest.mark.gpu

# fp32 parameters: with ns_steps = 0 the update (Frobenius norm lr) is a
# fraction of a bf16 spacing of the weights, so bf16 storage would hide it.
SPECS = [W.MuonSpec("a", 2, 128, 320, "f32", "f32", w_std=1.0, g_std=1.0),
         W.MuonSpec("b", 1, 300, 96, "f32", "bf16", w_std=0.5),
         W.MuonSpec("c", 1, 64, 64, "f32", "f32", w_std=0.5, g_std=0.3)]


@pytest.mark.parametrize("ns_steps", [0, 1, 2])
@pytest.mark.parametrize("flags", [dict(), dict(normuon=True), dict(muon_plus=True, cautious=1),
                                   dict(normuon=True, cautious=2),
                                   dict(normuon=True, muon_plus=True, cautious=2)])
def test_few_newton_schulz_steps(ns_steps, flags):
    wl = _wl(SPECS, ns_steps=ns_steps, **flags)
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check(wl, run)


def test_empty_tensors_are_skipped_beside_others():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    from tests.helpers import to_np
    import synth
    dev = "cuda"
    w = torch.tensor(synth.normal(95, 0, (256, 512), std=1.0), dtype=torch.float32, device=dev)
    g = torch.tensor(synth.normal(96, 0, (256, 512), std=1.0), dtype=torch.float32, device=dev)
    b = torch.zeros_like(w)
    e_w = torch.empty((0, 64), dtype=torch.float32, device=dev)
    e_g, e_b = torch.empty_like(e_w), torch.empty_like(e_w)
    w0 = w.clone()
    ts = [mh.muon_tensor(e_w, e_g, e_b, 1, None, 1.0, 0.01),
          mh.muon_tensor(w, g, b, 1, None, 1.0, 0.01),
          mh.muon_tensor(e_w, e_g, e_b, 1, None, 1.0, 0.01)]
    hp = mh.make_hparams()
    ws = torch.empty(mh.muon_workspace_bytes(ts, hp), dtype=torch.uint8, device=dev)
    mh.muon_step_batched(ts, hp, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    mh.workspace_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    from tests.parity import check_f32_update, check_fp32, momentum_atol
    res = oracle.muon_step_view(to_np(w0), to_np(g), np.zeros((256, 512)), oracle.MuonHparams(),
                                1.0, 0.01)
    check_fp32(to_np(b), res.B, momentum_atol(np.zeros((256, 512)), to_np(g), 0.95),
               "empty tensors beside: momentum")
    check_f32_update(to_np(w), res.W, (1 - 0.02 * 0.01) * to_np(w0), "empty tensors beside: param")


# Column counts that are not multiples of 8 take the tiled prologue (not the
# flat stream), scalar parameter access and ragged GEMM/statistics tiles.
RAGGED = [W.MuonSpec("r1", 3, 33, 65, "f32", "f32", w_std=1.0, g_std=1.0),
          W.MuonSpec("r2", 1, 130, 37, "f32", "bf16", w_std=0.5),
          W.MuonSpec("r3", 2, 57, 250, "f32", "f32", w_std=0.5, g_std=0.3),
          W.MuonSpec("r4", 1, 1, 77, "f32", "f32", w_std=1.0),
          W.MuonSpec("r5", 1, 77, 1, "f32", "f32", w_std=1.0)]


@pytest.mark.parametrize("flags", [dict(), dict(normuon=True), dict(muon_plus=True, cautious=1),
                                   dict(normuon=True, muon_plus=True, cautious=2)])
def test_ragged_shapes_full_step(flags):
    wl = _wl(RAGGED, steps=2, **flags)
    _run_and_check_last_step(wl, DeviceRun(wl), 2)


# bf16 parameters with fp32 gradients (and the reverse): the cautious-update
# mask reads the gradient in its own dtype, in the fused GEMM update and in
# the separate apply pass.
MIXED = [W.MuonSpec("m1", 1, 256, 512, "bf16", "f32", w_std=1.0, g_std=1.0),
         W.MuonSpec("m2", 2, 300, 128, "bf16", "f32", w_std=1.0, g_std=1.0),
         W.MuonSpec("m3", 1, 96, 200, "f32", "bf16", w_std=1.0, g_std=1.0),
         W.MuonSpec("m4", 1, 64, 100, "bf16", "bf16", w_std=0.02, g_std=1.0)]


@pytest.mark.parametrize("flags", [dict(cautious=2), dict(cautious=1),
                                   dict(normuon=True, cautious=2), dict(normuon=True),
                                   dict(normuon=True, muon_plus=True, cautious=1)])
def test_mixed_dtypes_with_cautious_masks(flags):
    wl = _wl(MIXED, **flags)
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check(wl, run)


# More tensors than one elementwise batch (64) and than one part of a
# streaming cautious-update launch (32): the parts count their tiles from their
# own first tile. Mixed shapes, views and parameter dtypes, bf16 gradients.
MANY = [W.MuonSpec(f"t{i}", 1 + i % 3, 64 + 32 * (i % 5), 256 + 64 * (i % 4),
                   "bf16" if i % 2 else "f32", "bf16",
                   w_std=0.02 if i % 2 else 1.0, g_std=1.0) for i in range(70)]


@pytest.mark.parametrize("flags", [dict(normuon=True, muon_plus=True, cautious=2),
                                   dict(normuon=True, cautious=1)])
def test_many_tensors_span_several_launches(flags):
    wl = _wl(MANY, **flags)
    run = DeviceRun(wl)
    run.step()
    run.status_ok()
    _check(wl, run)


# 63 one-tile tensors before one 4096 x 4096 view: 2111 tiles, so each of the
# 152 blocks of a streaming launch takes 14 consecutive tiles and the first
# blocks cross a tensor boundary at every tile. Their job records cycle through
# the ring of 4-8 slots several times (a slot is reused only once every tile
# of its tensor has been consumed). Every reduction runs in a fixed order, so
# the batched step must equal the same tensors stepped one call each, bit for
# bit; the large view is also checked against the oracle. (The 32 x 256 views
# are below the size where the bf16 iteration meets the 2e-2 bar: the
# bf16-storage model of it is 2.2-2.5 % off on them.)
RING = ([W.MuonSpec(f"s{i}", 1, 32, 256, "bf16", "bf16", w_std=0.02, g_std=1.0)
         for i in range(63)]
        + [W.MuonSpec("big", 1, 4096, 4096, "bf16", "bf16", w_std=0.02, g_std=1.0)])


@pytest.mark.parametrize("flags", [dict(normuon=True, muon_plus=True, cautious=2),
                                   dict(normuon=True, muon_plus=True, cautious=1)])
def test_job_ring_wraps_within_a_block(flags):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    wl = _wl(RING, **flags)
    batched = DeviceRun(wl)
    batched.step()
    batched.status_ok()
    single = DeviceRun(wl)
    stream = torch.cuda.current_stream().cuda_stream
    for t in single.ts:
        need = mh.muon_workspace_bytes([t], single.hp)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        mh.muon_step_batched([t], single.hp, ws.data_ptr(), need, stream)
        mh.workspace_status(ws.data_ptr(), stream)
    torch.cuda.synchronize()
    for i in range(len(RING)):
        assert torch.equal(batched.mW[i], single.mW[i]), ("parameter", i)
        assert torch.equal(batched.mB[i], single.mB[i]), ("momentum", i)
        assert torch.equal(batched.sm[i], single.sm[i]), ("NorMuon state", i)
    _check(wl, batched, tensors=[len(RING) - 1])
