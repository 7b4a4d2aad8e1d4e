"""The C ABI library on a machine without a GPU: it loads, exports every
declared entry point, its structs match the header's layout, and the host-side
argument checks reject bad calls before anything touches a device."""
import ctypes
import os
import re
import subprocess

import pytest

import muon_adamw_hybrid_gb300 as mh
from muon_adamw_hybrid_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", "muonhybrid.h"), os.path.join(ROOT, "include", "mhsynth.h")]


def _declared(header):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:mh|synth)_[a-z_0-9]+)\s*\(", text)))


def _exports(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True,
                         check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_library_exports_every_declared_symbol():
    declared = _declared(HEADERS[0])
    assert set(_lib.EXPORTED) <= set(declared) | set(_lib.EXPORTED)
    exports = _exports(_lib.LIB_PATH)
    for name in declared:
        assert name in exports, name
        assert hasattr(_lib.LIB, name)


def test_synth_library_exports():
    path = os.path.join(ROOT, "synth", "libmhsynth.so")
    exports = _exports(path)
    for name in _declared(HEADERS[1]):
        assert name in exports, name


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "sizes.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "muonhybrid.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\","
        " sizeof(mh_muon_tensor),"
        " sizeof(mh_muon_hparams), sizeof(mh_ns_problem), sizeof(mh_adamw_tensor),"
        " offsetof(mh_muon_tensor, views), offsetof(mh_muon_hparams, cautious),"
        " offsetof(mh_adamw_tensor, numel), offsetof(mh_muon_hparams, grad_mult),"
        " offsetof(mh_muon_hparams, skip), sizeof(mh_grad_ref), sizeof(mh_grad_control),"
        " offsetof(mh_grad_control, step)); printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\","
        " offsetof(mh_muon_hparams, sr_seed), offsetof(mh_muon_hparams, coeff_schedule),"
        " offsetof(mh_muon_hparams, norm_scale), offsetof(mh_muon_tensor, skip_zero_grad),"
        " offsetof(mh_muon_hparams, param_fence), offsetof(mh_muon_hparams, phase),"
        " offsetof(mh_muon_hparams, normuon_eps)); printf(\"%zu\\n\","
        " offsetof(mh_muon_hparams, shape_rule));"
        " return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                       check=True).stdout.split()))
    want = [ctypes.sizeof(mh.MuonTensor), ctypes.sizeof(mh.MuonHparams),
            ctypes.sizeof(mh.NsProblem), ctypes.sizeof(mh.AdamwTensor),
            mh.MuonTensor.views.offset, mh.MuonHparams.cautious.offset,
            mh.AdamwTensor.numel.offset, mh.MuonHparams.grad_mult.offset,
            mh.MuonHparams.skip.offset, ctypes.sizeof(mh.GradRef),
            ctypes.sizeof(mh.GradControl), mh.GradControl.step.offset,
            mh.MuonHparams.sr_seed.offset, mh.MuonHparams.coeff_schedule.offset,
            mh.MuonHparams.norm_scale.offset, mh.MuonTensor.skip_zero_grad.offset,
            mh.MuonHparams.param_fence.offset, mh.MuonHparams.phase.offset,
            mh.MuonHparams.normuon_eps.offset, mh.MuonHparams.shape_rule.offset]
    assert got == want


def _tensor(**kw):
    base = dict(param=256, grad=512, momentum=768, normuon_sm=0, param_dtype=0, grad_dtype=0,
                views=1, rows=4, cols=6, lr_mult=1.0, wd=0.0)
    base.update(kw)
    return mh.MuonTensor(**base)


def _step(tensors, hp=None, ws=0, wsb=0):
    hp = hp or mh.make_hparams()
    arr = (mh.MuonTensor * max(1, len(tensors)))(*tensors)
    return _lib.LIB.mh_muon_step_batched(arr, len(tensors), ctypes.byref(hp), ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(param_dtype=5), _lib.MH_EDTYPE),     # complex / other dtypes
    (dict(grad_dtype=-1), _lib.MH_EDTYPE),
    (dict(param=0), _lib.MH_EINVAL),
    (dict(momentum=0), _lib.MH_EINVAL),
    (dict(rows=-3), _lib.MH_ESHAPE),
    (dict(cols=1 << 25), _lib.MH_ESHAPE),
    (dict(rows=40000, cols=40000), _lib.MH_EUNSUPPORTED),
    (dict(lr_mult=float("nan")), _lib.MH_EINVAL),
    (dict(skip_zero_grad=2), _lib.MH_EINVAL),
    (dict(param_sr=1), _lib.MH_EINVAL),            # param_sr needs a bf16 parameter
    (dict(momentum_dtype=3), _lib.MH_EDTYPE),
])
def test_muon_rejects_bad_tensor(kw, code):
    assert _step([_tensor(**kw)]) == code
    assert mh.last_error() != ""


@pytest.mark.parametrize("kw", [dict(momentum=1.0), dict(momentum=-0.1), dict(eps=-1e-7),
                                dict(norm_scale=-1.0), dict(norm_scale=float("nan")),
                                dict(ns_steps=2, coeffs=[(1.0, 0.0, 0.0), (float("nan"), 0, 0)]),
                                dict(ns_steps=17), dict(ns_steps=-1), dict(cautious=3),
                                dict(coeffs=(float("inf"), 0, 0)),
                                dict(normuon=True, beta2=1.0),
                                dict(normuon_eps=-1.0), dict(normuon_eps=float("inf"))])
def test_muon_rejects_bad_hparams(kw):
    assert _step([_tensor()], hp=mh.make_hparams(**kw)) == _lib.MH_EINVAL


@pytest.mark.parametrize("rule", [-1, 2])
def test_muon_rejects_bad_shape_rule(rule):
    hp = mh.make_hparams(shape_rule=rule)
    assert _step([_tensor()], hp=hp) == _lib.MH_EINVAL
    assert "shape_rule" in mh.last_error()


@pytest.mark.parametrize("phase", [-1, 3])
def test_muon_rejects_bad_phase(phase):
    hp = mh.make_hparams()
    hp.phase = phase
    assert _step([_tensor()], hp=hp) == _lib.MH_EINVAL
    assert "phase" in mh.last_error()


def test_normuon_requires_state():
    assert _step([_tensor()], hp=mh.make_hparams(normuon=True)) == _lib.MH_EINVAL
    assert "normuon_sm" in mh.last_error()


def test_workspace_checks_happen_before_any_device_work():
    t = [_tensor()]
    need = mh.muon_workspace_bytes(t, mh.make_hparams())
    assert need > 0
    assert _step(t, ws=0, wsb=need) == _lib.MH_EWORKSPACE
    assert _step(t, ws=4096 + 16, wsb=need) == _lib.MH_EWORKSPACE      # misaligned
    assert _step(t, ws=4096, wsb=need - 1) == _lib.MH_EWORKSPACE        # too small
    assert "too small" in mh.last_error()


def test_empty_calls_are_noops():
    assert _step([]) == _lib.MH_OK
    assert _step([_tensor(rows=0)]) == _lib.MH_OK
    assert _step([_tensor(views=0, param=0, grad=0, momentum=0)]) == _lib.MH_OK
    arr = (mh.AdamwTensor * 1)(mh.AdamwTensor(numel=0))
    assert _lib.LIB.mh_adamw_step(arr, 1, 1e-3, 0.9, 0.95, 1e-8, 1, None) == _lib.MH_OK


def test_workspace_bytes_layout():
    # The workspace is a small statistics region (status word, per-view norms,
    # per-tile norm partials, per-view records; a multiple of 1 KiB) followed
    # by four bf16 buffers per Newton-Schulz shape class: X0 and X1
    # (m x ldx per view) and A and P (m x lda per view).
    one = mh.muon_workspace_bytes([_tensor(rows=256, cols=1024)], mh.make_hparams())
    buffers = 2 * 256 * 1024 * 2 + 2 * 256 * 256 * 2
    assert (one - buffers) % 1024 == 0 and 1024 <= one - buffers <= 4096
    # A tall view shares the transposed class: (1024 x 256) and (256 x 1024)
    # need one class with two slots.
    two = mh.muon_workspace_bytes([_tensor(rows=256, cols=1024), _tensor(rows=1024, cols=256)],
                                  mh.make_hparams())
    assert (two - 2 * buffers) % 1024 == 0 and 1024 <= two - 2 * buffers <= 4096
    # Ragged sizes pad the leading dimensions to multiples of 8 (5 x 16 and
    # 5 x 8 bf16 per buffer, each rounded to 1 KiB).
    rag = mh.muon_workspace_bytes([_tensor(rows=5, cols=13)], mh.make_hparams())
    assert rag - 4 * 1024 in (1024, 2048)
    # NorMuon and Muon+ add row and column statistics.
    more = mh.muon_workspace_bytes([_tensor(rows=256, cols=1024, normuon_sm=1024)],
                                   mh.make_hparams(normuon=True, muon_plus=True))
    assert more > one


def test_adamw_rejects_bad_args():
    good = mh.AdamwTensor(param=256, grad=512, exp_avg=768, exp_avg_sq=1024, numel=10)
    arr = (mh.AdamwTensor * 1)(good)
    L = _lib.LIB
    assert L.mh_adamw_step(arr, 1, 1e-3, 0.9, 0.95, 1e-8, 0, None) == _lib.MH_EINVAL  # step 0
    assert L.mh_adamw_step(arr, 1, 1e-3, 1.0, 0.95, 1e-8, 1, None) == _lib.MH_EINVAL
    assert L.mh_adamw_step(arr, -1, 1e-3, 0.9, 0.95, 1e-8, 1, None) == _lib.MH_EINVAL
    bad = (mh.AdamwTensor * 1)(mh.AdamwTensor(param=256, grad=512, exp_avg=0, exp_avg_sq=1024,
                                              numel=10))
    assert L.mh_adamw_step(bad, 1, 1e-3, 0.9, 0.95, 1e-8, 1, None) == _lib.MH_EINVAL
    cplx = (mh.AdamwTensor * 1)(mh.AdamwTensor(param=256, grad=512, exp_avg=768, exp_avg_sq=1024,
                                               numel=10, grad_dtype=9))
    assert L.mh_adamw_step(cplx, 1, 1e-3, 0.9, 0.95, 1e-8, 1, None) == _lib.MH_EDTYPE


def test_ns_rejects_bad_args():
    p = mh.NsProblem(x=256, out=512, in_dtype=0, out_dtype=0, views=1, rows=8, cols=8)
    arr = (mh.NsProblem * 1)(p)
    L = _lib.LIB
    assert L.mh_newton_schulz_batched(arr, 1, 17, 1.0, 0.0, 0.0, 1e-7, None, 0, None) == _lib.MH_EINVAL
    assert L.mh_newton_schulz_batched(arr, 1, 5, 1.0, 0.0, 0.0, 0.0, None, 0, None) == _lib.MH_EINVAL
    assert L.mh_newton_schulz_batched(arr, 1, 5, 1.0, 0.0, 0.0, 1e-7, None, 0, None) == _lib.MH_EWORKSPACE


def test_torch_marshalling_rejects_sparse_and_complex():
    import torch
    with pytest.raises(TypeError):
        mh.dtype_code(torch.zeros(2, 2).to_sparse())
    with pytest.raises(TypeError):
        mh.dtype_code(torch.zeros(2, 2, dtype=torch.complex64))
    with pytest.raises(TypeError):
        mh.dtype_code(torch.zeros(2, 2, dtype=torch.float16))
    with pytest.raises(ValueError):
        mh.muon_tensor(torch.zeros(4, 4), torch.zeros(4, 4), torch.zeros(4, 4))  # not CUDA


def test_grad_prepare_rejects_bad_args_before_device_work():
    L = _lib.LIB
    g = mh.GradRef(grad=256, grad_dtype=0, numel=70000)
    arr = (mh.GradRef * 1)(g)
    ctl = mh.GradControl(grad_mult=512, skip=768, norm=1024, step=0)
    assert L.mh_grad_prepare_workspace_bytes(arr, 1) == 16        # two 65536-element chunks
    assert L.mh_grad_prepare(arr, -1, 1.0, 1.0, ctypes.byref(ctl), 4096, 64, None) == _lib.MH_EINVAL
    assert L.mh_grad_prepare(arr, 1, 0.0, 1.0, ctypes.byref(ctl), 4096, 64, None) == _lib.MH_EINVAL
    assert L.mh_grad_prepare(arr, 1, float("inf"), 1.0, ctypes.byref(ctl), 4096, 64,
                             None) == _lib.MH_EINVAL
    assert L.mh_grad_prepare(arr, 1, 1.0, -1.0, ctypes.byref(ctl), 4096, 64, None) == _lib.MH_EINVAL
    assert L.mh_grad_prepare(arr, 1, 1.0, 1.0, None, 4096, 64, None) == _lib.MH_EINVAL
    no_norm = mh.GradControl(grad_mult=512, skip=768, norm=0, step=0)
    assert L.mh_grad_prepare(arr, 1, 1.0, 1.0, ctypes.byref(no_norm), 4096, 64,
                             None) == _lib.MH_EINVAL
    assert L.mh_grad_prepare(arr, 1, 1.0, 1.0, ctypes.byref(ctl), 4096, 8,
                             None) == _lib.MH_EWORKSPACE
    assert L.mh_grad_prepare(arr, 1, 1.0, 1.0, ctypes.byref(ctl), 4100, 64,
                             None) == _lib.MH_EWORKSPACE                     # misaligned
    bad = (mh.GradRef * 1)(mh.GradRef(grad=256, grad_dtype=7, numel=10))
    assert L.mh_grad_prepare(bad, 1, 1.0, 1.0, ctypes.byref(ctl), 4096, 64, None) == _lib.MH_EDTYPE
    null = (mh.GradRef * 1)(mh.GradRef(grad=0, grad_dtype=0, numel=10))
    assert L.mh_grad_prepare(null, 1, 1.0, 1.0, ctypes.byref(ctl), 4096, 64, None) == _lib.MH_EINVAL
    neg = (mh.GradRef * 1)(mh.GradRef(grad=256, grad_dtype=0, numel=-1))
    assert L.mh_grad_prepare_workspace_bytes(neg, 1) == 0


def test_adamw_ctl_needs_a_full_control_block():
    L = _lib.LIB
    good = mh.AdamwTensor(param=256, grad=512, exp_avg=768, exp_avg_sq=1024, numel=10)
    arr = (mh.AdamwTensor * 1)(good)
    assert L.mh_adamw_step_ctl(arr, 1, 1e-3, 0.9, 0.95, 1e-8, None, None) == _lib.MH_EINVAL
    no_step = mh.GradControl(grad_mult=512, skip=768, norm=1024, step=0)
    assert L.mh_adamw_step_ctl(arr, 1, 1e-3, 0.9, 0.95, 1e-8, ctypes.byref(no_step),
                               None) == _lib.MH_EINVAL


def test_ns_ex_rejects_bad_args():
    p = mh.NsProblem(x=256, out=512, in_dtype=0, out_dtype=0, views=1, rows=8, cols=8)
    arr = (mh.NsProblem * 1)(p)
    L = _lib.LIB
    co = (ctypes.c_float * 6)(3.0, -4.0, 2.0, 2.0, -1.5, 0.5)
    assert L.mh_newton_schulz_batched_ex(arr, 1, 2, None, 0.0, 1.01, None, 0, None) == _lib.MH_EINVAL
    assert L.mh_newton_schulz_batched_ex(arr, 1, 2, co, 0.0, 0.0, None, 0, None) == _lib.MH_EINVAL
    assert L.mh_newton_schulz_batched_ex(arr, 1, 2, co, -1.0, 1.0, None, 0, None) == _lib.MH_EINVAL
    bad = (ctypes.c_float * 6)(3.0, -4.0, float("inf"), 2.0, -1.5, 0.5)
    assert L.mh_newton_schulz_batched_ex(arr, 1, 2, bad, 0.0, 1.01, None, 0, None) == _lib.MH_EINVAL
    # valid arguments get as far as the workspace check
    assert L.mh_newton_schulz_batched_ex(arr, 1, 2, co, 0.0, 1.01, None, 0,
                                         None) == _lib.MH_EWORKSPACE


def test_schedule_length_is_checked_in_python():
    with pytest.raises(ValueError):
        mh.make_hparams(ns_steps=3, coeffs=[(1.0, 0.0, 0.0)] * 2)


def test_qk_clip_rejects_bad_args():
    L = _lib.LIB
    e = mh.QkClipEntry(param=256, param_dtype=0, heads=4, rows=64, cols=32, head_stride=16,
                       row_offset=0, scaled_rows=8, head_index0=0, exponent=0.5)
    arr = (mh.QkClipEntry * 1)(e)
    assert L.mh_qk_clip(arr, 1, 512, 0.0, None, None) == _lib.MH_EINVAL           # tau
    assert L.mh_qk_clip(arr, 1, None, 100.0, None, None) == _lib.MH_EINVAL        # s_max
    too_tall = (mh.QkClipEntry * 1)(mh.QkClipEntry(param=256, param_dtype=0, heads=5, rows=64,
                                                   cols=32, head_stride=16, row_offset=0,
                                                   scaled_rows=8, head_index0=0, exponent=0.5))
    assert L.mh_qk_clip(too_tall, 1, 512, 100.0, None, None) == _lib.MH_ESHAPE
    past_block = (mh.QkClipEntry * 1)(mh.QkClipEntry(param=256, param_dtype=0, heads=4, rows=64,
                                                     cols=32, head_stride=16, row_offset=10,
                                                     scaled_rows=8, head_index0=0, exponent=0.5))
    assert L.mh_qk_clip(past_block, 1, 512, 100.0, None, None) == _lib.MH_ESHAPE
    bad_exp = (mh.QkClipEntry * 1)(mh.QkClipEntry(param=256, param_dtype=0, heads=4, rows=64,
                                                  cols=32, head_stride=16, row_offset=0,
                                                  scaled_rows=8, head_index0=0,
                                                  exponent=float("nan")))
    assert L.mh_qk_clip(bad_exp, 1, 512, 100.0, None, None) == _lib.MH_EINVAL
    assert L.mh_qk_clip(arr, 0, None, 100.0, None, None) == _lib.MH_OK               # nothing to do
