"""The inactive-expert rule on the GPU against the oracle (kimi-k3
"Optimization", "One more kind of state: which experts learn?": a routed
expert that received no gradient acquires no momentum and no weight decay).

A flagged view whose gradient is zero everywhere must come back bit for bit
unchanged (parameter, momentum, NorMuon state); every other view follows the
usual bars (tests.parity: momentum element by element against the running
bound on fp32 rounding; the fp32 parameter by its update, within the
Newton-Schulz bar; NorMuon state 3e-2).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import rel_fro, to_np
from tests.parity import check_f32_update, check_fp32, momentum_atol

pytestmark = pytest.mark.gpu

# name, views, rows, cols, flagged, silent views
SPECS = [("e0.gate_up", 2, 96, 128, True, (0,)),      # one silent view of two
         ("e1.down", 1, 128, 96, True, (0,)),         # tall, silent
         ("e2.big", 1, 1408, 2048, True, (0,)),       # silent over many chunks
         ("e3.gate_up", 2, 96, 128, True, ()),        # active expert
         ("dense", 1, 128, 128, False, (0,))]         # silent but not flagged: it moves


def _run(hp_kw):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    hp = mh.make_hparams(**hp_kw)
    tens, keep = [], []
    for t, (name, views, r, c, flag, silent) in enumerate(SPECS):
        w = synth.normal(80, t, (views * r, c), std=1.0).astype(np.float64)
        g = synth.normal(81, t, (views * r, c), std=1e-3).astype(np.float64)
        b = synth.normal(82, t, (views * r, c), std=1e-3).astype(np.float64)
        for v in silent:
            g[v * r:(v + 1) * r] = 0.0
        dw = torch.tensor(w, dtype=torch.float32, device="cuda")
        dg = torch.tensor(g, dtype=torch.float32, device="cuda")
        db = torch.tensor(b, dtype=torch.float32, device="cuda")
        sm = (torch.full((views * r,), 0.25, dtype=torch.float32, device="cuda")
              if hp_kw.get("normuon") else None)
        keep.append(dict(w=w, g=g, b=b, dw=dw, dg=dg, db=db, sm=sm))
        tens.append(mh.muon_tensor(dw, dg, db, views, sm, 1.0, 0.01, skip_zero_grad=flag))
    ws = torch.empty(mh.muon_workspace_bytes(tens, hp), dtype=torch.uint8, device="cuda")
    mh.muon_step_batched(tens, hp, ws.data_ptr(), ws.numel(),
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    mh.workspace_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return keep


@pytest.mark.parametrize("hp_kw", [dict(), dict(normuon=True), dict(cautious=1),
                                   dict(muon_plus=True), dict(normuon=True, muon_plus=True,
                                                              cautious=2)])
def test_inactive_views_are_untouched_and_the_rest_match(hp_kw):
    keep = _run(hp_kw)
    ohp = oracle.MuonHparams(normuon=hp_kw.get("normuon", False),
                             muon_plus=hp_kw.get("muon_plus", False),
                             cautious=hp_kw.get("cautious", 0))
    for (name, views, r, c, flag, silent), k in zip(SPECS, keep):
        W0 = k["w"].astype(np.float32).astype(np.float64)
        sm0 = None if k["sm"] is None else np.full(views * r, 0.25)
        Wn, Bn, _, smn = oracle.muon_step_tensor(W0, k["g"], k["b"], ohp, views=views, wd=0.01,
                                                 sm=sm0, skip_zero_grad=flag)
        got_w = to_np(k["dw"])
        got_b = to_np(k["db"])
        for v in range(views):
            rows = slice(v * r, (v + 1) * r)
            if flag and v in silent:
                np.testing.assert_array_equal(got_w[rows], W0[rows], err_msg=name)
                np.testing.assert_array_equal(got_b[rows], k["b"][rows].astype(np.float32),
                                              err_msg=name)
                if k["sm"] is not None:
                    assert np.all(to_np(k["sm"])[rows] == 0.25), name
                continue
            b0 = k["b"][rows].astype(np.float32).astype(np.float64)
            check_fp32(got_b[rows], Bn[rows], momentum_atol(b0, k["g"][rows], 0.95),
                       f"experts {name}[{v}] momentum")
            base = W0[rows] if ohp.cautious else 0.9998 * W0[rows]
            check_f32_update(got_w[rows], Wn[rows], base, f"experts {name}[{v}]")
            if k["sm"] is not None:
                assert rel_fro(to_np(k["sm"])[rows], smn.reshape(-1)[rows]) < 3e-2, (name, v)
    # the unflagged silent tensor did move (decay and momentum), unless the
    # cautious-update mask is on: it keeps only entries whose update agrees
    # with a gradient that is zero everywhere here
    dense = keep[-1]
    moved = not np.array_equal(to_np(dense["dw"]), dense["w"].astype(np.float32))
    assert moved == (hp_kw.get("cautious", 0) != 2)
