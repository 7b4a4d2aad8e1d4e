"""The allocation-free Newton-Schulz entry point (mh_newton_schulz_batched_noalloc).

It exists for callers that cannot allocate device memory or keep a scratch
buffer of their own (a plugin given only its input and output buffers, a
program whose device memory is all reserved by its own pool). Its scratch is
a fixed 64 MiB array inside the library. These tests call it through the C
ABI and compare it with the regular entry point, which takes a workspace
from the caller. Both run the same kernels with reductions in a fixed order,
so the results must be identical bit for bit. Two calls in a row use
different problem lists (a larger matrix first, then ragged smaller ones
whose column counts are not multiples of 8), so the second call's plan lays
the shared array out differently from the first: anything the first call
left behind that the second read would show up as a difference.

This file is named to be collected last.
"""

import pytest

import synth
from muon_adamw_hybrid_gb300 import _lib

COEFFS = (3.4445, -4.7750, 2.0315)


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


SHAPE_LISTS = {
    # one larger matrix first (about 29 MiB of scratch) ...
    "large": [((1536, 3072), 1, "f32"), ((2 * 256, 512), 2, "bf16")],
    # ... then ragged smaller ones, cols not multiples of 8, tall and wide
    "ragged": [((300, 203), 1, "f32"), ((3 * 97, 61), 3, "bf16"), ((129, 517), 1, "bf16"),
               ((256, 768), 1, "f32")],
}


_LAST = []


def _run_both(seed, shapes):
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    stream = torch.cuda.current_stream().cuda_stream
    xs = [torch.tensor(synth.normal(seed, k, s), device="cuda").to(tdt[dt])
          for k, (s, _, dt) in enumerate(shapes)]
    views = [v for _, v, _ in shapes]
    # Regular entry point, caller-provided workspace.
    ref = [torch.full_like(x, float("nan")) for x in xs]
    arr, n = _problems(xs, ref, views)
    need = _lib.LIB.mh_ns_workspace_bytes(arr, n)
    assert 0 < need <= _lib.NS_STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = _lib.LIB.mh_newton_schulz_batched(arr, n, 5, *COEFFS, 1e-7, ws.data_ptr(), need, stream)
    assert rc == _lib.MH_OK, _lib.last_error()
    # Allocation-free entry point, same problems, no workspace argument.
    got = [torch.full_like(x, float("nan")) for x in xs]
    arr2, n2 = _problems(xs, got, views)
    rc = _lib.LIB.mh_newton_schulz_batched_noalloc(arr2, n2, 5, *COEFFS, 1e-7, stream)
    assert rc == _lib.MH_OK, _lib.last_error()
    torch.cuda.synchronize()
    return [(g.cpu(), r.cpu()) for g, r in zip(got, ref)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    # Two calls in a row with different problem lists (and so different
    # scratch layouts); each must equal the workspace entry point exactly.
    for seed, key in ((101, "large"), (202, "ragged")):
        _LAST[:] = _run_both(seed, SHAPE_LISTS[key])
        for got, ref in _LAST:
            assert torch.isfinite(got.float()).all()
            # bit for bit: compare the raw storage, so -0.0 / +0.0 would differ too
            g = got.view(torch.int16 if got.dtype == torch.bfloat16 else torch.int32)
            r = ref.view(torch.int16 if ref.dtype == torch.bfloat16 else torch.int32)
            assert torch.equal(g, r), (key, tuple(got.shape))
        # and, as a sanity check, each result is a Newton-Schulz output: its
        # squared singular values average near one.
        for (s, v, _), (got, _) in zip(SHAPE_LISTS[key], _LAST):
            r, c = s[0] // v, s[1]
            ms = float(got.double().pow(2).sum()) / (v * min(r, c))
            assert 0.3 < ms < 1.5, (key, s, ms)


def test_noalloc_rejects_oversized_request_without_touching_the_device():
    # 4096 x 8192 needs far more than 64 MiB; the check happens on the host
    # before anything is enqueued (pointers are never dereferenced).
    p = _lib.NsProblem(x=256, out=512, in_dtype=0, out_dtype=0, views=1, rows=4096, cols=8192)
    arr = (_lib.NsProblem * 1)(p)
    rc = _lib.LIB.mh_newton_schulz_batched_noalloc(arr, 1, 5, *COEFFS, 1e-7, None)
    assert rc == _lib.MH_EWORKSPACE
    assert str(_lib.NS_STATIC_SCRATCH_BYTES) in _lib.last_error()
