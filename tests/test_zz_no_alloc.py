"""The allocation-free Newton-Schulz entry point (mh_newton_schulz_batched_noalloc).

It exists for callers that cannot allocate device memory or keep a scratch
buffer of their own (a plugin given only its input and output buffers, a
program whose device memory is all reserved by its own pool). Its scratch is
a fixed 64 MiB array inside the library. These tests call it through the C
ABI and compare it with the regular entry point, which takes a workspace
from the caller, within the Newton-Schulz tolerance the other tests use
(2e-2 relative Frobenius), on two calls in a row so that whatever the first
call left in the shared array cannot leak into the second.

This file is named to be collected last.
"""

import numpy as np
import pytest

import synth
from muon_adamw_hybrid_gb300 import _lib

COEFFS = (3.4445, -4.7750, 2.0315)
NS_TOL = 2e-2


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _problems(xs, outs, views):
    import torch
    probs = []
    for x, o, v in zip(xs, outs, views):
        dt = {torch.float32: _lib.MH_F32, torch.bfloat16: _lib.MH_BF16}
        probs.append(_lib.NsProblem(x=x.data_ptr(), out=o.data_ptr(), in_dtype=dt[x.dtype],
                                    out_dtype=dt[o.dtype], views=v, rows=x.shape[0] // v,
                                    cols=x.shape[1]))
    arr = (_lib.NsProblem * len(probs))(*probs)
    return arr, len(probs)


def _run_both(seed):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    shapes = [((256, 768), 1, torch.float32), ((2 * 384, 128), 2, torch.bfloat16),
              ((300, 200), 1, torch.float32)]
    xs = [torch.tensor(synth.normal(seed, k, s), device="cuda").to(dt)
          for k, (s, _, dt) in enumerate(shapes)]
    views = [v for _, v, _ in shapes]
    # Regular entry point, caller-provided workspace.
    ref = [torch.full_like(x, float("nan")) for x in xs]
    arr, n = _problems(xs, ref, views)
    need = _lib.LIB.mh_ns_workspace_bytes(arr, n)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = _lib.LIB.mh_newton_schulz_batched(arr, n, 5, *COEFFS, 1e-7, ws.data_ptr(), need, stream)
    assert rc == _lib.MH_OK, _lib.last_error()
    # Allocation-free entry point, same problems, no workspace argument.
    got = [torch.full_like(x, float("nan")) for x in xs]
    arr2, n2 = _problems(xs, got, views)
    rc = _lib.LIB.mh_newton_schulz_batched_noalloc(arr2, n2, 5, *COEFFS, 1e-7, stream)
    assert rc == _lib.MH_OK, _lib.last_error()
    torch.cuda.synchronize()
    return [(g.double().cpu().numpy(), r.double().cpu().numpy()) for g, r in zip(got, ref)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    for seed in (101, 202):  # two calls in a row, different inputs
        for got, ref in _run_both(seed):
            assert np.all(np.isfinite(got))
            assert _rel(got, ref) < NS_TOL


def test_noalloc_rejects_oversized_request_without_touching_the_device():
    # 4096 x 8192 needs far more than 64 MiB; the check happens on the host
    # before anything is enqueued (pointers are never dereferenced).
    p = _lib.NsProblem(x=256, out=512, in_dtype=0, out_dtype=0, views=1, rows=4096, cols=8192)
    arr = (_lib.NsProblem * 1)(p)
    rc = _lib.LIB.mh_newton_schulz_batched_noalloc(arr, 1, 5, *COEFFS, 1e-7, None)
    assert rc == _lib.MH_EWORKSPACE
    assert str(_lib.NS_STATIC_SCRATCH_BYTES) in _lib.last_error()
