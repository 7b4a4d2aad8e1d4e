"""fp64 CPU oracle of the AdamW half of the hybrid step.

TEST INFRASTRUCTURE ONLY; the product path never imports it.

The pages name AdamW without printing it (dew.training.optim, "OPTIMIZER_MAP":
optax.adamw; Speedtronic "v2 optimizers", "CPU/CUDA/MPS behavior": PyTorch's
fused AdamW). The reading used is the standard decoupled AdamW of those two
libraries: bias-corrected first and second moments, eps added outside the
square root, weight decay multiplied by the learning rate and applied to the
pre-update weight, step count t starting at 1.
"""
from __future__ import annotations

import numpy as np


def adamw_step(W, G, m, v, lr: float, beta1: float, beta2: float, eps: float,
               wd: float, step: int):
    """One AdamW step in float64. Returns (W_new, m_new, v_new)."""
    W = np.asarray(W, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m_new = beta1 * m + (1.0 - beta1) * G
    v_new = beta2 * v + (1.0 - beta2) * G * G
    m_hat = m_new / (1.0 - beta1 ** step)
    v_hat = v_new / (1.0 - beta2 ** step)
    W_new = W * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return W_new, m_new, v_new
