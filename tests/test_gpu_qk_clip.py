"""QK-Clip on the GPU against the oracle (kimi-k3 "Optimization", "QK-Clip
watches a different failure mode"; dew.training.optim "scale_by_qk_clip").

Rows of heads at or below tau must come back bit for bit; clipped rows match
the fp64 oracle to fp32 rounding (fp32 weights) or to one bf16 spacing (bf16
weights, where the factor's last bits can move a rounding)."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import to_np

pytestmark = pytest.mark.gpu

H, D, DM = 8, 16, 72


def _dev(x, dtype):
    import torch
    t = torch.tensor(np.asarray(x), dtype=torch.float64, device="cuda")
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


def _check(got, W0, entry, s, tau, dtype):
    want = oracle.qk_clip(W0, entry, s, tau)
    g = oracle.gamma(s, tau)
    for h in range(entry.heads):
        r0 = h * entry.head_stride + entry.row_offset
        rows = slice(r0, r0 + entry.scaled_rows)
        if g[entry.head_index0 + h] == 1.0:
            np.testing.assert_array_equal(got[rows], W0[rows])
        elif dtype == "f32":
            np.testing.assert_allclose(got[rows], want[rows], rtol=1e-6, atol=0)
        else:
            want_b = oracle.round_bf16(want[rows])
            np.testing.assert_allclose(got[rows], want_b, rtol=2.0 ** -7, atol=0)
    # rows outside every scaled block are untouched
    mask = np.ones(W0.shape[0], dtype=bool)
    for h in range(entry.heads):
        r0 = h * entry.head_stride + entry.row_offset
        mask[r0:r0 + entry.scaled_rows] = False
    np.testing.assert_array_equal(got[mask], W0[mask])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [DM, 69])             # 69: the unaligned, scalar path
def test_qk_clip_matches_oracle(dtype, cols):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    s = np.array([50, 150, 90, 400, 101, 99, 1000, 100], dtype=np.float32).astype(np.float64)
    tau = 100.0
    Wq = synth.normal(90, 1, (H * D, cols), dtype=dtype).astype(np.float64)
    Wkv = synth.normal(90, 2, (H * (D + 24), cols), dtype=dtype).astype(np.float64)  # K then V
    Wqb = synth.normal(90, 3, (H * (D + 8), cols), dtype=dtype).astype(np.float64)   # nope, rope
    dq, dkv, dqb = _dev(Wq, dtype), _dev(Wkv, dtype), _dev(Wqb, dtype)
    entries = [oracle.ClipEntry(H, D, 0, D, 0, 0.5),            # q_proj
               oracle.ClipEntry(H, D + 24, 0, D, 0, 0.5),       # kv_b_proj: K rows only
               oracle.ClipEntry(H, D + 8, 0, D, 0, 0.5),        # q_b_proj nope rows
               oracle.ClipEntry(H, D + 8, D, 8, 0, 1.0)]        # q_b_proj rope rows
    weights = [dq, dkv, dqb, dqb]
    ents = [mh.qk_clip_entry(w, e.heads, e.head_stride, e.scaled_rows, e.row_offset,
                             e.head_index0, e.exponent) for w, e in zip(weights, entries)]
    s_dev = torch.tensor(s, dtype=torch.float32, device="cuda")
    mh.qk_clip(ents, s_dev, tau)
    torch.cuda.synchronize()
    _check(to_np(dq), Wq, entries[0], s, tau, dtype)
    _check(to_np(dkv), Wkv, entries[1], s, tau, dtype)
    got_qb = to_np(dqb)
    want_qb = oracle.qk_clip(oracle.qk_clip(Wqb, entries[2], s, tau), entries[3], s, tau)
    tol = 1e-6 if dtype == "f32" else 2.0 ** -7
    np.testing.assert_allclose(got_qb, oracle.round_bf16(want_qb) if dtype == "bf16" else want_qb,
                               rtol=tol, atol=0)


def test_qk_clip_after_a_skipped_step_changes_nothing():
    import torch
    import muon_adamw_hybrid_gb300 as mh
    W = synth.normal(91, 1, (H * D, DM)).astype(np.float64)
    dw = _dev(W, "f32")
    ctl = mh.GradientControl("cuda")
    ctl.skip.fill_(1)
    s_dev = torch.full((H,), 1000.0, dtype=torch.float32, device="cuda")
    mh.qk_clip([mh.qk_clip_entry(dw, H, D, D)], s_dev, 100.0, control=ctl)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(dw), W.astype(np.float32))
    ctl.skip.fill_(0)
    mh.qk_clip([mh.qk_clip_entry(dw, H, D, D)], s_dev, 100.0, control=ctl)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(dw), W * np.sqrt(0.1), rtol=1e-6)
