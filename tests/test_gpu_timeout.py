"""The bounded-wait failure path of the Newton-Schulz GEMM stages and of the
streaming apply / column-statistics passes, on the GPU.

Every wait of a GEMM stage gives up after mh_set_wait_limit cycles; the
launch then records MH_ETIMEOUT in the workspace status word, lets the copies
and MMAs it issued land, frees its tensor memory and returns. With a limit of
2000 cycles (about a microsecond) the epilogue cannot wait out the first
block of a 4096-deep contraction (64 k-steps of MMAs, some tens of
microseconds), so the call must report the timeout; nothing faults, traps or
waits without a bound. With the default restored,
the same call on the same workspace then succeeds and matches the oracle, so
the context stays usable. A whole NorMuon + Muon+ step (GEMM stages and the
streaming passes, whose waits take the same limit) is run the same way, with
its state put back before the clean step.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import rel_fro, to_np

COEFFS = (3.4445, -4.7750, 2.0315)


def test_wait_limit_setter_rejects_negative_and_restores_default():
    from muon_adamw_hybrid_gb300 import _lib
    default = _lib.get_wait_limit()
    assert default > 10 ** 9
    assert _lib.LIB.mh_set_wait_limit(-1) == _lib.MH_EINVAL
    assert _lib.get_wait_limit() == default
    _lib.set_wait_limit(12345)
    assert _lib.get_wait_limit() == 12345
    _lib.set_wait_limit(0)
    assert _lib.get_wait_limit() == default


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1024, 4096), (4096, 1024)])
def test_short_wait_limit_times_out_then_a_normal_call_succeeds(shape):
    import torch
    import muon_adamw_hybrid_gb300 as mh
    from muon_adamw_hybrid_gb300 import _lib
    q = synth.normal(61, shape[0], shape).astype(np.float64)
    x = torch.tensor(q, dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x)
    probs = [mh.ns_problem(x, out, 1)]
    need = _lib.ns_workspace_bytes(probs)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    default = _lib.get_wait_limit()
    try:
        _lib.set_wait_limit(2000)
        mh.newton_schulz_batched(probs, 5, *COEFFS, 1e-7, ws.data_ptr(), need, stream)
        rc = _lib.LIB.mh_workspace_status(ws.data_ptr(), stream)
        assert rc == _lib.MH_ETIMEOUT, (rc, _lib.last_error())
    finally:
        _lib.set_wait_limit(0)
    assert _lib.get_wait_limit() == default
    torch.cuda.synchronize()
    # The same call again with the default limit: clean status, right answer.
    mh.newton_schulz_batched(probs, 5, *COEFFS, 1e-7, ws.data_ptr(), need, stream)
    mh.workspace_status(ws.data_ptr(), stream)
    torch.cuda.synchronize()
    assert rel_fro(to_np(out), oracle.newton_schulz(q)) < 2e-2


@pytest.mark.gpu
def test_short_wait_limit_in_a_full_step_then_a_clean_step():
    import torch
    from muon_adamw_hybrid_gb300 import _lib
    from synth import workloads as W
    from tests.helpers import DeviceRun
    from tests.test_gpu_muon import _check, _wl
    wl = _wl([W.MuonSpec("t", 2, 1024, 4096, "bf16", "bf16")], normuon=True, muon_plus=True,
             cautious=1)
    run = DeviceRun(wl)
    state = run.mW + run.mB + [s for s in run.sm if s is not None]
    saved = [t.clone() for t in state]
    stream = torch.cuda.current_stream().cuda_stream
    try:
        _lib.set_wait_limit(2000)
        run.step()
        rc = _lib.LIB.mh_workspace_status(run.ws.data_ptr(), stream)
        assert rc == _lib.MH_ETIMEOUT, (rc, _lib.last_error())
    finally:
        _lib.set_wait_limit(0)
    torch.cuda.synchronize()
    for t, c in zip(state, saved):
        t.copy_(c)
    run.step_count = 0
    run.step()
    run.status_ok()
    torch.cuda.synchronize()
    _check(wl, run)
