"""Non-finite inputs without gradient control: a NaN in one gradient entry
spoils exactly what the arithmetic says it spoils and nothing else.

Muon: the momentum is NaN at that entry only; the view's Newton-Schulz input is
normalised by a NaN norm, so that view's whole update and parameter are NaN;
every other view and tensor matches the oracle. AdamW: that element's
parameter and moments are NaN, every other element matches the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import to_np
from tests.parity import adamw_atol, check_f32_update, check_fp32, momentum_atol

pytestmark = pytest.mark.gpu


def test_muon_nan_gradient_stays_in_its_view():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    shapes = [(2, 128, 256), (1, 192, 64)]
    keep, ts = [], []
    for t, (v, r, c) in enumerate(shapes):
        w = synth.normal(70, t, (v * r, c), std=1.0).astype(np.float64)
        g = synth.normal(71, t, (v * r, c), std=1.0).astype(np.float64)
        if t == 0:
            g[r + 5, 17] = np.nan                     # view 1 of tensor 0
        dw = torch.tensor(w, dtype=torch.float32, device="cuda")
        dg = torch.tensor(g, dtype=torch.float32, device="cuda")
        db = torch.zeros_like(dw)
        keep.append((w, g, dw, dg, db))
        ts.append(mh.muon_tensor(dw, dg, db, v, None, 1.0, 0.01))
    hp = mh.make_hparams()
    ws = torch.empty(mh.muon_workspace_bytes(ts, hp), dtype=torch.uint8, device="cuda")
    mh.muon_step_batched(ts, hp, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    mh.workspace_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)

    ohp = oracle.MuonHparams()
    for t, ((v, r, c), (w, g, dw, dg, db)) in enumerate(zip(shapes, keep)):
        got_w, got_b = to_np(dw), to_np(db)
        for view in range(v):
            rows = slice(view * r, (view + 1) * r)
            if t == 0 and view == 1:
                assert np.isnan(got_w[rows]).all()
                nan_b = np.isnan(got_b[rows])
                assert nan_b.sum() == 1 and nan_b[5, 17]
                continue
            w32 = w[rows].astype(np.float32).astype(np.float64)
            res = oracle.muon_step_view(w32, g[rows], np.zeros((r, c)), ohp, 1.0, 0.01)
            check_fp32(got_b[rows], res.B, momentum_atol(np.zeros((r, c)), g[rows], 0.95),
                       f"nonfinite neighbour {t}[{view}] momentum")
            check_f32_update(got_w[rows], res.W, 0.9998 * w32, f"nonfinite neighbour {t}[{view}]")


def test_adamw_nan_gradient_stays_in_its_element():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    n = 10007
    w = synth.normal(72, 0, (n,), std=0.02).astype(np.float64)
    g = synth.normal(73, 0, (n,), std=1e-3).astype(np.float64)
    g[4321] = np.nan
    dw = torch.tensor(w, dtype=torch.float32, device="cuda")
    dg = torch.tensor(g, dtype=torch.float32, device="cuda")
    dm, dv = torch.zeros_like(dw), torch.zeros_like(dw)
    mh.adamw_step([mh.adamw_tensor(dw, dg, dm, dv, 1.0, 0.1)], 1e-3, 0.9, 0.95, 1e-8, 1,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    gw, gm, gv = to_np(dw), to_np(dm), to_np(dv)
    for arr in (gw, gm, gv):
        assert np.isnan(arr[4321]) and np.isnan(arr).sum() == 1
    ok = np.ones(n, bool)
    ok[4321] = False
    w32 = w.astype(np.float32).astype(np.float64)[ok]
    z = np.zeros(ok.sum())
    Wn, M, V = oracle.adamw_step(w32, g[ok], z, z, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    Em, Ev, Ew = adamw_atol(w32, g[ok], z, z, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    check_fp32(gm[ok], M, Em, "adamw beside a NaN: m")
    check_fp32(gv[ok], V, Ev, "adamw beside a NaN: v")
    check_fp32(gw[ok], Wn.astype(np.float32).astype(np.float64), Ew, "adamw beside a NaN: W")
