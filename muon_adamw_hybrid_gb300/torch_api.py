"""Marshalling from torch tensors to the C ABI, and an optimizer facade.

PyTorch supplies device memory and streams; every arithmetic step of the
optimizer runs in libmuonhybrid's kernels.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (MH_BF16, MH_F32, AdamwTensor, GradControl, GradRef, MuonHparams, MuonTensor,
                   NsProblem, QkClipEntry)

# Speedtronic docs "v2 optimizers", "Newton-Schulz": coefficients, steps, eps.
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
NS_EPS = 1e-7


def dtype_code(t: torch.Tensor) -> int:
    """fp32 -> MH_F32, bf16 -> MH_BF16; sparse, complex and other dtypes raise."""
    if t.layout != torch.strided:
        raise TypeError(f"sparse tensors are not supported (layout {t.layout})")
    if t.is_complex():
        raise TypeError(f"complex tensors are not supported (dtype {t.dtype})")
    if t.dtype == torch.float32:
        return MH_F32
    if t.dtype == torch.bfloat16:
        return MH_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: only float32 and bfloat16")


def _dev_ptr(t: torch.Tensor, what: str) -> int:
    """Device address of a tensor: a CUDA tensor, or a page-locked host
    tensor that the device reads in place (the kernels then stream it over
    the host link instead of a separate copy)."""
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.is_cuda:
        return t.data_ptr()
    if t.is_pinned() and _lib.pointer_device_accessible(t.data_ptr()):
        return t.data_ptr()
    raise ValueError(f"{what} must be a CUDA tensor or device-accessible pinned host memory")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _keep(struct, *tensors):
    """The C structs hold raw device pointers: the struct object keeps the
    tensors it points into alive for as long as it lives."""
    struct._tensors = tuple(t for t in tensors if t is not None)
    return struct


def make_hparams(lr=0.02, momentum=0.95, nesterov=True, eps=NS_EPS, ns_steps=NS_STEPS,
                 coeffs=NS_COEFFS, normuon=False, beta2=0.95, muon_plus=False, plus_eps=NS_EPS,
                 cautious=0, norm_scale=1.0, normuon_eps=1e-10, shape_rule=0) -> MuonHparams:
    """Muon hyperparameters. ``coeffs`` is one (a, b, c) for every iteration, or
    a sequence of ``ns_steps`` triples (flaxchat's Polar Express schedule);
    ``norm_scale`` gives X0 = Q / (||Q|| * norm_scale + eps); ``shape_rule``
    picks the update's shape factor (MH_SHAPE_RATIO or MH_SHAPE_MOONLIGHT)."""
    sched = None
    if len(coeffs) and not isinstance(coeffs[0], (int, float)):
        if len(coeffs) != ns_steps:
            raise ValueError(f"the schedule has {len(coeffs)} triples for {ns_steps} steps")
        flat = [float(v) for t in coeffs for v in t]
        sched = (ctypes.c_float * len(flat))(*flat)
        a, b, c = coeffs[0]
    else:
        a, b, c = coeffs
    hp = MuonHparams(lr=lr, momentum=momentum, nesterov=int(bool(nesterov)), eps=eps,
                     ns_steps=ns_steps, a=a, b=b, c=c, normuon=int(bool(normuon)), beta2=beta2,
                     muon_plus=int(bool(muon_plus)), plus_eps=plus_eps, cautious=int(cautious),
                     norm_scale=norm_scale, normuon_eps=normuon_eps,
                     shape_rule=int(shape_rule))
    if sched is not None:
        hp.coeff_schedule = ctypes.addressof(sched)
        hp._sched = sched          # the library reads it during each call
    return hp


def _view_dims(param: torch.Tensor, views: int, rows: int | None = None):
    if param.dim() < 2:
        raise ValueError("a Muon parameter must have at least 2 dimensions")
    cols = param.shape[-1]
    numel = param.numel()
    if rows is None:
        if views < 1 or numel % (views * cols):
            raise ValueError(f"shape {tuple(param.shape)} cannot be split into {views} views")
        rows = numel // (views * cols)
    if views * rows * cols != numel:
        raise ValueError(f"views*rows*cols != numel for shape {tuple(param.shape)}")
    return views, rows, cols


def muon_tensor(param: torch.Tensor, grad: torch.Tensor, momentum: torch.Tensor, views: int = 1,
                normuon_sm: torch.Tensor | None = None, lr_mult: float = 1.0,
                wd: float = 0.0, rows: int | None = None, param_sr: bool = False,
                skip_zero_grad: bool = False) -> MuonTensor:
    """One Muon-routed tensor: ``views`` independent matrices of rows x cols.

    ``param`` is (views*rows, cols) or (views, rows, cols), contiguous. The
    momentum buffer is float32, or bfloat16 (kept stochastically rounded);
    ``param_sr`` writes a bf16 parameter stochastically rounded;
    ``skip_zero_grad`` (routed experts) leaves a view whose gradient is zero
    everywhere untouched.
    """
    v, r, c = _view_dims(param, views, rows)
    if grad.numel() != param.numel() or momentum.numel() != param.numel():
        raise ValueError("grad and momentum must have the parameter's number of elements")
    sm = 0
    if normuon_sm is not None:
        if normuon_sm.dtype != torch.float32 or normuon_sm.numel() != v * r:
            raise ValueError("normuon_sm must be float32 with views*rows elements")
        sm = _dev_ptr(normuon_sm, "normuon_sm")
    st = MuonTensor(param=_dev_ptr(param, "param"), grad=_dev_ptr(grad, "grad"),
                    momentum=_dev_ptr(momentum, "momentum"), normuon_sm=sm,
                    param_dtype=dtype_code(param), grad_dtype=dtype_code(grad), views=v,
                    rows=r, cols=c, lr_mult=lr_mult, wd=wd, momentum_dtype=dtype_code(momentum),
                    param_sr=int(bool(param_sr)), skip_zero_grad=int(bool(skip_zero_grad)))
    return _keep(st, param, grad, momentum, normuon_sm)


def adamw_tensor(param, grad, exp_avg, exp_avg_sq, lr_mult: float = 1.0,
                 wd: float = 0.0, param_sr: bool = False) -> AdamwTensor:
    """One AdamW tensor; moments float32, or bfloat16 (kept stochastically
    rounded), both of one dtype."""
    n = param.numel()
    if grad.numel() != n or exp_avg.numel() != n or exp_avg_sq.numel() != n:
        raise ValueError("grad and moments must have the parameter's number of elements")
    if exp_avg.dtype != exp_avg_sq.dtype:
        raise TypeError("both AdamW moments must have one dtype")
    st = AdamwTensor(param=_dev_ptr(param, "param"), grad=_dev_ptr(grad, "grad"),
                     exp_avg=_dev_ptr(exp_avg, "exp_avg"),
                     exp_avg_sq=_dev_ptr(exp_avg_sq, "exp_avg_sq"),
                     param_dtype=dtype_code(param), grad_dtype=dtype_code(grad), numel=n,
                     lr_mult=lr_mult, wd=wd, state_dtype=dtype_code(exp_avg),
                     param_sr=int(bool(param_sr)))
    return _keep(st, param, grad, exp_avg, exp_avg_sq)


def ns_problem(x: torch.Tensor, out: torch.Tensor, views: int = 1) -> NsProblem:
    v, r, c = _view_dims(x, views)
    if out.numel() != x.numel():
        raise ValueError("out must have x's number of elements")
    st = NsProblem(x=_dev_ptr(x, "x"), out=_dev_ptr(out, "out"), in_dtype=dtype_code(x),
                   out_dtype=dtype_code(out), views=v, rows=r, cols=c)
    return _keep(st, x, out)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Caller-owned workspace (PyTorch allocations are 512-byte aligned)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def newton_schulz(xs, outs=None, views=None, steps: int = NS_STEPS, coeffs=NS_COEFFS,
                  eps: float = NS_EPS, workspace: torch.Tensor | None = None, stream=None,
                  norm_scale: float = 1.0):
    """U = NS(X) for a list of matrices (or stacks of views); returns the outputs.
    ``coeffs``: one (a, b, c), or ``steps`` of them (one per iteration)."""
    xs = list(xs)
    if outs is None:
        outs = [torch.empty_like(x) for x in xs]
    views = views or [1] * len(xs)
    probs = [ns_problem(x, o, v) for x, o, v in zip(xs, outs, views)]
    need = _lib.ns_workspace_bytes(probs)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, xs[0].device)
    if len(coeffs) and not isinstance(coeffs[0], (int, float)):
        if len(coeffs) != steps:
            raise ValueError(f"the schedule has {len(coeffs)} triples for {steps} steps")
        _lib.newton_schulz_batched_ex(probs, list(coeffs), eps, norm_scale, workspace.data_ptr(),
                                      workspace.numel(), _stream_ptr(stream))
    elif norm_scale != 1.0:
        _lib.newton_schulz_batched_ex(probs, [tuple(coeffs)] * steps, eps, norm_scale,
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_ptr(stream))
    else:
        a, b, c = coeffs
        _lib.newton_schulz_batched(probs, steps, a, b, c, eps, workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(stream))
    return outs


def grad_ref(g: torch.Tensor) -> GradRef:
    return _keep(GradRef(grad=_dev_ptr(g, "grad"), grad_dtype=dtype_code(g), numel=g.numel()), g)


class GradientControl:
    """Device-resident result of grad_prepare, read by the step kernels.

    kimi-k3 "Optimization", "Keep the arithmetic and gradients under control":
    one global gradient norm over both groups, a clip when max_norm > 0, and
    the whole hybrid update skipped when an unscaled gradient is inf or NaN.
    ``grad_mult`` (float32), ``skip`` (int32), ``norm`` (float64) and ``step``
    (int64, the count of applied steps, used for AdamW's bias correction) are
    one-element device tensors.
    """

    def __init__(self, device, step: int = 0):
        self.grad_mult = torch.ones(1, dtype=torch.float32, device=device)
        self.skip = torch.zeros(1, dtype=torch.int32, device=device)
        self.norm = torch.zeros(1, dtype=torch.float64, device=device)
        self.step = torch.full((1,), int(step), dtype=torch.int64, device=device)

    def struct(self) -> GradControl:
        return GradControl(grad_mult=self.grad_mult.data_ptr(), skip=self.skip.data_ptr(),
                           norm=self.norm.data_ptr(), step=self.step.data_ptr())


def grad_prepare(grads, control: GradientControl, inv_loss_scale: float = 1.0,
                 max_norm: float = 0.0, workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Global norm, clip factor and overflow skip of ``grads`` into ``control``
    (all on the device, stream-ordered). Returns the workspace it used."""
    refs = [grad_ref(g) for g in grads]
    need = _lib.grad_prepare_workspace_bytes(refs)
    if workspace is None or workspace.numel() < need:
        workspace = alloc_workspace(need, control.norm.device)
    _lib.grad_prepare(refs, inv_loss_scale, max_norm, control.struct(), workspace.data_ptr(),
                      workspace.numel(), _stream_ptr(stream))
    return workspace


def qk_clip_entry(param: torch.Tensor, heads: int, head_stride: int, scaled_rows: int,
                  row_offset: int = 0, head_index0: int = 0,
                  exponent: float = 0.5) -> QkClipEntry:
    """Rows of a (rows, cols) query / key projection that QK-Clip rescales:
    for each of ``heads`` blocks of ``head_stride`` rows, ``scaled_rows`` rows
    from ``row_offset`` are multiplied by gamma_h ** exponent."""
    if param.dim() != 2:
        raise ValueError("a QK-Clip entry names a 2-D weight")
    st = QkClipEntry(param=_dev_ptr(param, "param"), param_dtype=dtype_code(param), heads=heads,
                     rows=param.shape[0], cols=param.shape[1], head_stride=head_stride,
                     row_offset=row_offset, scaled_rows=scaled_rows, head_index0=head_index0,
                     exponent=exponent)
    return _keep(st, param)


def qk_clip(entries, s_max: torch.Tensor, tau: float = 100.0,
            control: "GradientControl | None" = None, stream=None) -> None:
    """kimi-k3 "QK-Clip" / dew "scale_by_qk_clip": rescale the listed rows of
    every head with s_max[h] > tau by (tau / s_max[h]) ** exponent, after the
    optimizer update; nothing happens after a step the control block skipped."""
    if s_max.dtype != torch.float32:
        raise TypeError("s_max must be float32")
    skip = control.skip.data_ptr() if control is not None else None
    _lib.qk_clip(list(entries), _dev_ptr(s_max, "s_max"), tau, skip, _stream_ptr(stream))


@dataclass
class MuonGroupEntry:
    param: torch.Tensor
    views: int = 1
    lr_mult: float = 1.0
    wd: float = 0.0
    skip_zero_grad: bool = False   # routed experts: no momentum or decay without gradient


@dataclass
class AdamGroupEntry:
    param: torch.Tensor
    lr_mult: float = 1.0
    wd: float = 0.0


class HybridMuonAdamW:
    """Owns the optimizer state of a hybrid Muon + AdamW step and calls the library.

    Muon state: one fp32 momentum buffer per routed tensor (views share it),
    plus the NorMuon second moment when enabled. AdamW state: fp32 exp_avg and
    exp_avg_sq. The state dict holds exactly these tensors and the AdamW step
    count (Speedtronic "Scheduler and checkpoint behavior": Adam moments and
    Muon momentum buffers; the cautious variants add no state).
    """

    def __init__(self, muon_params, adamw_params, lr=0.02, momentum=0.95, nesterov=True,
                 ns_steps=NS_STEPS, coeffs=NS_COEFFS, eps=NS_EPS, normuon=False,
                 normuon_beta2=0.95, muon_plus=False, plus_eps=NS_EPS, cautious=0,
                 adam_lr=3e-4, adam_betas=(0.9, 0.95), adam_eps=1e-8, max_grad_norm=None,
                 state_dtype=torch.float32, param_sr=False, normuon_eps=1e-10, shape_rule=0):
        self.muon = [e if isinstance(e, MuonGroupEntry) else MuonGroupEntry(**e) for e in muon_params]
        self.adam = [e if isinstance(e, AdamGroupEntry) else AdamGroupEntry(**e) for e in adamw_params]
        self.hp = make_hparams(lr, momentum, nesterov, eps, ns_steps, coeffs, normuon,
                               normuon_beta2, muon_plus, plus_eps, cautious,
                               normuon_eps=normuon_eps, shape_rule=shape_rule)
        self.adam_lr, self.adam_betas, self.adam_eps = adam_lr, adam_betas, adam_eps
        self.step_count = 0
        # dew.training.optim "bf16_moments": bf16 state is kept stochastically
        # rounded; param_sr does the same for bf16 parameters.
        if state_dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("state_dtype must be torch.float32 or torch.bfloat16")
        self.param_sr = bool(param_sr)
        self.momentum = [torch.zeros(e.param.shape, dtype=state_dtype, device=e.param.device)
                         for e in self.muon]
        self.normuon_sm = []
        for e in self.muon:
            if normuon:
                v, r, _ = _view_dims(e.param, e.views)
                self.normuon_sm.append(torch.zeros(v * r, dtype=torch.float32, device=e.param.device))
            else:
                self.normuon_sm.append(None)
        self.exp_avg = [torch.zeros(e.param.shape, dtype=state_dtype, device=e.param.device)
                        for e in self.adam]
        self.exp_avg_sq = [torch.zeros_like(m) for m in self.exp_avg]
        self._ws = None
        # Gradient control (global norm / clip / overflow skip), on when
        # max_grad_norm is given (0 = observe the norm without clipping).
        self.max_grad_norm = max_grad_norm
        self.control = None
        self._gws = None
        if max_grad_norm is not None:
            dev = (self.muon or self.adam)[0].param.device
            self.control = GradientControl(dev)
            self.hp.grad_mult = self.control.grad_mult.data_ptr()
            self.hp.skip = self.control.skip.data_ptr()

    @property
    def lr(self) -> float:
        return self.hp.lr

    @lr.setter
    def lr(self, value: float) -> None:
        self.hp.lr = value

    def _muon_structs(self, grads):
        return [muon_tensor(e.param, g, m, e.views, sm, e.lr_mult, e.wd,
                            param_sr=self.param_sr and e.param.dtype == torch.bfloat16,
                            skip_zero_grad=e.skip_zero_grad)
                for e, g, m, sm in zip(self.muon, grads, self.momentum, self.normuon_sm)]

    def _adam_structs(self, grads):
        return [adamw_tensor(e.param, g, m, v, e.lr_mult, e.wd,
                             param_sr=self.param_sr and e.param.dtype == torch.bfloat16)
                for e, g, m, v in zip(self.adam, grads, self.exp_avg, self.exp_avg_sq)]

    def workspace_bytes(self) -> int:
        return _lib.muon_workspace_bytes(self._muon_structs([e.param for e in self.muon]), self.hp)

    def step(self, muon_grads=None, adam_grads=None, stream=None,
             inv_loss_scale: float = 1.0, param_fence=None) -> None:
        """One hybrid step. Gradients default to each parameter's ``.grad``.

        With gradient control on, the gradients are first unscaled by
        ``inv_loss_scale``, their global norm is taken and clipped to
        ``max_grad_norm``, and the whole step is skipped on the device when one
        of them is inf or NaN (``self.control.skip``); no host sync happens.

        ``param_fence`` (a recorded ``torch.cuda.Event``): the step's stream
        waits for it just before the first kernel that writes a parameter, so
        work ordered before it on another stream (a copy of the previous
        step's parameters) overlaps the momentum and Newton-Schulz kernels."""
        muon_grads = muon_grads if muon_grads is not None else [e.param.grad for e in self.muon]
        adam_grads = adam_grads if adam_grads is not None else [e.param.grad for e in self.adam]
        s = _stream_ptr(stream)
        if self.control is not None:
            self._gws = grad_prepare(list(muon_grads) + list(adam_grads), self.control,
                                     inv_loss_scale, float(self.max_grad_norm), self._gws, stream)
        elif inv_loss_scale != 1.0:
            raise ValueError("inv_loss_scale needs gradient control (pass max_grad_norm)")
        self.step_count += 1
        self.hp.sr_seed = self.step_count   # a fresh rounding stream every call
        if self.muon:
            ts = self._muon_structs(muon_grads)
            need = _lib.muon_workspace_bytes(ts, self.hp)
            if self._ws is None or self._ws.numel() < need:
                self._ws = alloc_workspace(need, self.muon[0].param.device)
            self.hp.param_fence = param_fence.cuda_event if param_fence is not None else None
            try:
                _lib.muon_step_batched(ts, self.hp, self._ws.data_ptr(), self._ws.numel(), s)
            finally:
                self.hp.param_fence = None
        elif param_fence is not None:
            (stream or torch.cuda.current_stream()).wait_event(param_fence)
        if self.adam:
            b1, b2 = self.adam_betas
            if self.control is not None:
                _lib.adamw_step_ctl(self._adam_structs(adam_grads), self.adam_lr, b1, b2,
                                    self.adam_eps, self.control.struct(), s)
            else:
                _lib.adamw_step(self._adam_structs(adam_grads), self.adam_lr, b1, b2,
                                self.adam_eps, self.step_count, s)

    def applied_steps(self) -> int:
        """Steps actually applied (skipped ones excluded when gradient control is on)."""
        if self.control is not None:
            return int(self.control.step.item())
        return self.step_count

    def state_dict(self) -> dict:
        return {"step": self.applied_steps(),
                "momentum": [m.clone() for m in self.momentum],
                "normuon_sm": [None if s is None else s.clone() for s in self.normuon_sm],
                "exp_avg": [m.clone() for m in self.exp_avg],
                "exp_avg_sq": [v.clone() for v in self.exp_avg_sq]}

    def load_state_dict(self, sd: dict) -> None:
        self.step_count = int(sd["step"])
        if self.control is not None:
            self.control.step.fill_(self.step_count)
        for dst, src in zip(self.momentum, sd["momentum"]):
            dst.copy_(src)
        for dst, src in zip(self.normuon_sm, sd["normuon_sm"]):
            if dst is not None:
                dst.copy_(src)
        for dst, src in zip(self.exp_avg, sd["exp_avg"]):
            dst.copy_(src)
        for dst, src in zip(self.exp_avg_sq, sd["exp_avg_sq"]):
            dst.copy_(src)
