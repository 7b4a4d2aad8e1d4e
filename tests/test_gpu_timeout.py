"""The bounded-wait failure path of the Newton-Schulz GEMM stages, on the GPU.

Every wait of a GEMM stage gives up after mh_set_wait_limit cycles; the
launch then records MH_ETIMEOUT in the workspace status word, lets the copies
and MMAs it issued land, frees its tensor memory and returns. With a limit of
2000 cycles (about a microsecond) the epilogue cannot wait out the first
block of a 4096-deep contraction (64 k-steps of MMAs, some tens of
microseconds), so the call must report the timeout; nothing faults, traps or
waits without a bound. With the default restored,
the same call on the same workspace then succeeds and matches the oracle, so
the context stays usable.
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
