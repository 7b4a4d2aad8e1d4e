"""fp64 CPU oracle of the gradient control ahead of both halves of the step.

TEST INFRASTRUCTURE ONLY; the product path never imports it.

Sources (page title, section):
  [KIMI] kimi-k3, "Optimization", "Keep the arithmetic and gradients under
         control": before the optimizer step the trainer measures the global
         gradient norm; a positive max_grad_norm clips it when needed, 0
         disables clipping while the norm is still observed; FP16 training
         uses a gradient scaler, and an overflow skips the whole hybrid
         update, not only the Muon half.
  [DEW]  dew.training.optim, "build_optimizer": the global-norm clip reads
         every gradient together, before the parameter groups split them.

Readings taken where the pages are silent (each also listed in the design
notes):
  * The norm is the L2 norm over every element of every gradient of both
    groups, taken of the unscaled gradient g * inv_loss_scale.
  * "Clips that norm if necessary": every gradient is multiplied by
    min(1, max_norm / (norm + 1e-6)), PyTorch's clip_grad_norm_ definition
    (the trainer on that page is a PyTorch one; optax's clip_by_global_norm
    differs only in the 1e-6 guard).
  * "Overflow": some unscaled gradient element is inf or NaN. The step then
    writes nothing (no momentum, moment, NorMuon state or parameter) and the
    step count used for bias correction does not advance.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

CLIP_EPS = 1e-6


@dataclass
class GradControl:
    norm: float    # global norm of the unscaled gradients (observed even without clipping)
    mult: float    # factor every raw gradient element is multiplied by (0 when skipping)
    skip: bool     # an unscaled gradient element was inf or NaN


def grad_control(grads, inv_loss_scale: float = 1.0, max_norm: float = 0.0) -> GradControl:
    """[KIMI] + [DEW]: one global norm over all gradients, then the clip
    factor, or the skip decision."""
    total = 0.0
    finite = True
    for g in grads:
        u = np.asarray(g, dtype=np.float64).ravel() * inv_loss_scale
        if not np.all(np.isfinite(u)):
            finite = False
            continue
        total += float(np.dot(u, u))
    if not finite:
        return GradControl(norm=math.nan, mult=0.0, skip=True)
    norm = math.sqrt(total)
    coef = 1.0
    if max_norm > 0.0:
        coef = min(1.0, max_norm / (norm + CLIP_EPS))
    return GradControl(norm=norm, mult=inv_loss_scale * coef, skip=False)
