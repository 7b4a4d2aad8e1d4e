"""ctypes binding of libmuonhybrid (include/muonhybrid.h): argument marshalling only.

Every computation runs in the CUDA library. If the library has not been built
the import fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64,
                    c_void_p)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmuonhybrid.so")

MH_OK, MH_EINVAL, MH_EDTYPE, MH_ESHAPE, MH_EWORKSPACE, MH_ECUDA, MH_EUNSUPPORTED, MH_ETIMEOUT = range(8)
STATUS_NAMES = {0: "MH_OK", 1: "MH_EINVAL", 2: "MH_EDTYPE", 3: "MH_ESHAPE", 4: "MH_EWORKSPACE",
                5: "MH_ECUDA", 6: "MH_EUNSUPPORTED", 7: "MH_ETIMEOUT"}
MH_F32, MH_BF16 = 0, 1
MH_CAUTIOUS_OFF, MH_CAUTIOUS_WD, MH_CAUTIOUS_UPDATE = 0, 1, 2
MH_STEP_ALL, MH_STEP_GRADIENTS, MH_STEP_FINISH = 0, 1, 2
MH_SHAPE_RATIO, MH_SHAPE_MOONLIGHT = 0, 1

EXPORTED = ("mh_muon_workspace_bytes", "mh_muon_step_batched", "mh_ns_workspace_bytes",
            "mh_newton_schulz_batched", "mh_adamw_step", "mh_workspace_status", "mh_last_error",
            "mh_version", "mh_profiler_enable", "mh_profiler_reset", "mh_profiler_read",
            "mh_newton_schulz_batched_noalloc", "mh_grad_prepare_workspace_bytes",
            "mh_grad_prepare", "mh_adamw_step_ctl", "mh_newton_schulz_batched_ex", "mh_qk_clip",
            "mh_pointer_device_accessible", "mh_set_wait_limit", "mh_get_wait_limit")
NS_STATIC_SCRATCH_BYTES = 64 << 20


class MuonTensor(ctypes.Structure):
    _fields_ = [("param", c_void_p), ("grad", c_void_p), ("momentum", c_void_p),
                ("normuon_sm", c_void_p), ("param_dtype", c_int32), ("grad_dtype", c_int32),
                ("views", c_int64), ("rows", c_int64), ("cols", c_int64),
                ("lr_mult", c_float), ("wd", c_float), ("momentum_dtype", c_int32),
                ("param_sr", c_int32), ("skip_zero_grad", c_int32)]


class MuonHparams(ctypes.Structure):
    _fields_ = [("lr", c_float), ("momentum", c_float), ("nesterov", c_int32), ("eps", c_float),
                ("ns_steps", c_int32), ("a", c_float), ("b", c_float), ("c", c_float),
                ("normuon", c_int32), ("beta2", c_float), ("muon_plus", c_int32),
                ("plus_eps", c_float), ("cautious", c_int32),
                ("grad_mult", c_void_p), ("skip", c_void_p), ("sr_seed", c_uint64),
                ("coeff_schedule", c_void_p), ("norm_scale", c_float),
                ("param_fence", c_void_p), ("phase", c_int32), ("normuon_eps", c_float),
                ("shape_rule", c_int32)]


class NsProblem(ctypes.Structure):
    _fields_ = [("x", c_void_p), ("out", c_void_p), ("in_dtype", c_int32), ("out_dtype", c_int32),
                ("views", c_int64), ("rows", c_int64), ("cols", c_int64)]


class AdamwTensor(ctypes.Structure):
    _fields_ = [("param", c_void_p), ("grad", c_void_p), ("exp_avg", c_void_p),
                ("exp_avg_sq", c_void_p), ("param_dtype", c_int32), ("grad_dtype", c_int32),
                ("numel", c_int64), ("lr_mult", c_float), ("wd", c_float),
                ("state_dtype", c_int32), ("param_sr", c_int32)]


class GradRef(ctypes.Structure):
    _fields_ = [("grad", c_void_p), ("grad_dtype", c_int32), ("numel", c_int64)]


class GradControl(ctypes.Structure):
    _fields_ = [("grad_mult", c_void_p), ("skip", c_void_p), ("norm", c_void_p),
                ("step", c_void_p)]


class QkClipEntry(ctypes.Structure):
    _fields_ = [("param", c_void_p), ("param_dtype", c_int32), ("heads", c_int32),
                ("rows", c_int64), ("cols", c_int64), ("head_stride", c_int64),
                ("row_offset", c_int64), ("scaled_rows", c_int64), ("head_index0", c_int32),
                ("exponent", c_float)]


class KernelStats(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", c_int64), ("total_ms", ctypes.c_double),
                ("bytes", ctypes.c_double), ("flops", ctypes.c_double),
                ("flops_executed", ctypes.c_double)]


class MuonHybridError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python muon_adamw_hybrid_gb300/build.py, or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    lib.mh_muon_workspace_bytes.argtypes = [POINTER(MuonTensor), c_int32, POINTER(MuonHparams)]
    lib.mh_muon_workspace_bytes.restype = c_size_t
    lib.mh_muon_step_batched.argtypes = [POINTER(MuonTensor), c_int32, POINTER(MuonHparams),
                                         c_void_p, c_size_t, c_void_p]
    lib.mh_muon_step_batched.restype = c_int
    lib.mh_ns_workspace_bytes.argtypes = [POINTER(NsProblem), c_int32]
    lib.mh_ns_workspace_bytes.restype = c_size_t
    lib.mh_newton_schulz_batched.argtypes = [POINTER(NsProblem), c_int32, c_int32, c_float,
                                             c_float, c_float, c_float, c_void_p, c_size_t,
                                             c_void_p]
    lib.mh_newton_schulz_batched.restype = c_int
    lib.mh_newton_schulz_batched_ex.argtypes = [POINTER(NsProblem), c_int32, c_int32,
                                                POINTER(c_float), c_float, c_float, c_void_p,
                                                c_size_t, c_void_p]
    lib.mh_newton_schulz_batched_ex.restype = c_int
    lib.mh_newton_schulz_batched_noalloc.argtypes = [POINTER(NsProblem), c_int32, c_int32,
                                                     c_float, c_float, c_float, c_float, c_void_p]
    lib.mh_newton_schulz_batched_noalloc.restype = c_int
    lib.mh_adamw_step.argtypes = [POINTER(AdamwTensor), c_int32, c_float, c_float, c_float,
                                  c_float, c_int64, c_void_p]
    lib.mh_adamw_step.restype = c_int
    lib.mh_adamw_step_ctl.argtypes = [POINTER(AdamwTensor), c_int32, c_float, c_float, c_float,
                                      c_float, POINTER(GradControl), c_void_p]
    lib.mh_adamw_step_ctl.restype = c_int
    lib.mh_grad_prepare_workspace_bytes.argtypes = [POINTER(GradRef), c_int32]
    lib.mh_grad_prepare_workspace_bytes.restype = c_size_t
    lib.mh_grad_prepare.argtypes = [POINTER(GradRef), c_int32, c_float, c_float,
                                    POINTER(GradControl), c_void_p, c_size_t, c_void_p]
    lib.mh_grad_prepare.restype = c_int
    lib.mh_qk_clip.argtypes = [POINTER(QkClipEntry), c_int32, c_void_p, c_float, c_void_p,
                               c_void_p]
    lib.mh_qk_clip.restype = c_int
    lib.mh_pointer_device_accessible.argtypes = [c_void_p, POINTER(c_int32)]
    lib.mh_pointer_device_accessible.restype = c_int
    lib.mh_workspace_status.argtypes = [c_void_p, c_void_p]
    lib.mh_workspace_status.restype = c_int
    lib.mh_set_wait_limit.argtypes = [c_int64]
    lib.mh_set_wait_limit.restype = c_int
    lib.mh_get_wait_limit.argtypes = []
    lib.mh_get_wait_limit.restype = c_int64
    lib.mh_last_error.argtypes = []
    lib.mh_last_error.restype = c_char_p
    lib.mh_version.argtypes = []
    lib.mh_version.restype = c_char_p
    lib.mh_profiler_enable.argtypes = [c_int32]
    lib.mh_profiler_enable.restype = c_int
    lib.mh_profiler_reset.argtypes = []
    lib.mh_profiler_reset.restype = c_int
    lib.mh_profiler_read.argtypes = [POINTER(KernelStats), c_int32, POINTER(c_int32)]
    lib.mh_profiler_read.restype = c_int
    return lib


LIB = _load()


def last_error() -> str:
    return LIB.mh_last_error().decode()


def version() -> str:
    return LIB.mh_version().decode()


def _check(status: int) -> None:
    if status != MH_OK:
        raise MuonHybridError(status, last_error())


def _array(struct, items):
    n = len(items)
    arr = (struct * max(n, 1))(*items)
    return arr, n


def muon_workspace_bytes(tensors, hparams: MuonHparams) -> int:
    arr, n = _array(MuonTensor, tensors)
    nbytes = LIB.mh_muon_workspace_bytes(arr, n, ctypes.byref(hparams))
    if nbytes == 0 and n > 0 and last_error():
        raise MuonHybridError(MH_EINVAL, last_error())
    return int(nbytes)


def muon_step_batched(tensors, hparams: MuonHparams, workspace: int, workspace_bytes: int,
                      stream: int) -> None:
    arr, n = _array(MuonTensor, tensors)
    _check(LIB.mh_muon_step_batched(arr, n, ctypes.byref(hparams), workspace, workspace_bytes,
                                    stream))


def ns_workspace_bytes(problems) -> int:
    arr, n = _array(NsProblem, problems)
    return int(LIB.mh_ns_workspace_bytes(arr, n))


def newton_schulz_batched(problems, steps: int, a: float, b: float, c: float, eps: float,
                          workspace: int, workspace_bytes: int, stream: int) -> None:
    arr, n = _array(NsProblem, problems)
    _check(LIB.mh_newton_schulz_batched(arr, n, steps, a, b, c, eps, workspace, workspace_bytes,
                                        stream))


def newton_schulz_batched_ex(problems, coeffs, eps: float, norm_scale: float, workspace: int,
                             workspace_bytes: int, stream: int) -> None:
    """Newton-Schulz with one (a, b, c) per iteration (a sequence of triples)
    and the normalisation X0 / (||X0|| * norm_scale + eps)."""
    arr, n = _array(NsProblem, problems)
    flat = [float(v) for t in coeffs for v in t]
    carr = (c_float * max(len(flat), 1))(*flat)
    _check(LIB.mh_newton_schulz_batched_ex(arr, n, len(coeffs), carr, eps, norm_scale, workspace,
                                           workspace_bytes, stream))


def newton_schulz_batched_noalloc(problems, steps: int, a: float, b: float, c: float, eps: float,
                                  stream: int) -> None:
    """mh_newton_schulz_batched without a workspace argument: the scratch is a
    fixed 64 MiB array inside the library, for callers that cannot allocate."""
    arr, n = _array(NsProblem, problems)
    _check(LIB.mh_newton_schulz_batched_noalloc(arr, n, steps, a, b, c, eps, stream))


def adamw_step(tensors, lr: float, beta1: float, beta2: float, eps: float, step: int,
               stream: int) -> None:
    arr, n = _array(AdamwTensor, tensors)
    _check(LIB.mh_adamw_step(arr, n, lr, beta1, beta2, eps, step, stream))


def adamw_step_ctl(tensors, lr: float, beta1: float, beta2: float, eps: float,
                   control: GradControl, stream: int) -> None:
    arr, n = _array(AdamwTensor, tensors)
    _check(LIB.mh_adamw_step_ctl(arr, n, lr, beta1, beta2, eps, ctypes.byref(control), stream))


def grad_prepare_workspace_bytes(grads) -> int:
    arr, n = _array(GradRef, grads)
    nbytes = LIB.mh_grad_prepare_workspace_bytes(arr, n)
    if nbytes == 0:
        raise MuonHybridError(MH_EINVAL, last_error())
    return int(nbytes)


def grad_prepare(grads, inv_loss_scale: float, max_norm: float, control: GradControl,
                 workspace: int, workspace_bytes: int, stream: int) -> None:
    arr, n = _array(GradRef, grads)
    _check(LIB.mh_grad_prepare(arr, n, inv_loss_scale, max_norm, ctypes.byref(control),
                               workspace, workspace_bytes, stream))


def qk_clip(entries, s_max: int, tau: float, skip: int, stream: int) -> None:
    arr, n = _array(QkClipEntry, entries)
    _check(LIB.mh_qk_clip(arr, n, s_max, tau, skip, stream))


def pointer_device_accessible(ptr: int) -> bool:
    """True when the current device reads and writes ``ptr`` at that address
    (device or managed memory, or mapped page-locked host memory)."""
    out = c_int32(0)
    _check(LIB.mh_pointer_device_accessible(ptr, ctypes.byref(out)))
    return bool(out.value)


def workspace_status(workspace: int, stream: int) -> None:
    _check(LIB.mh_workspace_status(workspace, stream))


def set_wait_limit(cycles: int) -> None:
    """Bounded-wait limit of the GEMM stages in SM cycles (0: the default)."""
    _check(LIB.mh_set_wait_limit(int(cycles)))


def get_wait_limit() -> int:
    return int(LIB.mh_get_wait_limit())


def profiler_enable(on: bool = True) -> None:
    _check(LIB.mh_profiler_enable(1 if on else 0))


def profiler_reset() -> None:
    _check(LIB.mh_profiler_reset())


def profiler_read() -> dict:
    """Per kernel family: launches, total_ms, bytes, flops, flops_executed."""
    cap = 64
    arr = (KernelStats * cap)()
    n = c_int32(0)
    _check(LIB.mh_profiler_read(arr, cap, ctypes.byref(n)))
    out = {}
    for k in range(min(n.value, cap)):
        r = arr[k]
        out[r.name.decode()] = dict(launches=int(r.launches), total_ms=float(r.total_ms),
                                    bytes=float(r.bytes), flops=float(r.flops),
                                    flops_executed=float(r.flops_executed))
    return out
