"""GB300-native hybrid Muon + AdamW optimizer step.

The computation lives in ``libmuonhybrid.so`` (CUDA for sm_103a, C ABI in
include/muonhybrid.h). This package is a thin binding:

* ``_lib``      ctypes structures and the C entry points, one to one;
* ``torch_api`` marshalling from torch tensors (device memory and streams
  come from PyTorch) and a small optimizer facade that owns the state;
* ``routing``   the host-side Muon/AdamW parameter split (not on the step's
  hot path).

Importing the package loads the library and raises if it is missing.
"""
from ._lib import (MH_BF16, MH_CAUTIOUS_OFF, MH_CAUTIOUS_UPDATE, MH_CAUTIOUS_WD, MH_F32,
                   MH_SHAPE_MOONLIGHT, MH_SHAPE_RATIO, MH_STEP_ALL, MH_STEP_FINISH,
                   MH_STEP_GRADIENTS,
                   AdamwTensor, GradControl, GradRef, MuonHparams, MuonHybridError, MuonTensor,
                   NsProblem, QkClipEntry, adamw_step, adamw_step_ctl,
                   grad_prepare_workspace_bytes,
                   last_error, muon_step_batched, muon_workspace_bytes, newton_schulz_batched,
                   ns_workspace_bytes, pointer_device_accessible, profiler_enable, profiler_read,
                   profiler_reset, version, workspace_status)
from .torch_api import (GradientControl, HybridMuonAdamW, adamw_tensor, dtype_code, grad_prepare,
                        grad_ref, make_hparams, muon_tensor, newton_schulz, ns_problem, qk_clip,
                        qk_clip_entry)
from .routing import route_parameters

__all__ = [
    "MH_BF16", "MH_CAUTIOUS_OFF", "MH_CAUTIOUS_UPDATE", "MH_CAUTIOUS_WD", "MH_F32",
    "MH_SHAPE_MOONLIGHT", "MH_SHAPE_RATIO", "MH_STEP_ALL", "MH_STEP_FINISH", "MH_STEP_GRADIENTS",
    "AdamwTensor",
    "GradControl", "GradRef", "MuonHparams", "MuonHybridError", "MuonTensor", "NsProblem",
    "adamw_step", "adamw_step_ctl", "grad_prepare_workspace_bytes", "last_error",
    "muon_step_batched", "muon_workspace_bytes", "newton_schulz_batched", "ns_workspace_bytes",
    "version", "workspace_status", "profiler_enable", "profiler_read", "profiler_reset",
    "GradientControl", "HybridMuonAdamW", "adamw_tensor", "dtype_code", "grad_prepare",
    "grad_ref", "make_hparams", "muon_tensor", "newton_schulz", "ns_problem", "route_parameters",
    "QkClipEntry", "qk_clip", "qk_clip_entry", "pointer_device_accessible",
]
