"""Pins for the oracle's AdamW (CPU only): PyTorch's own AdamW in float64,
and the step-1 closed form."""
import numpy as np
import pytest
import torch

import oracle
import synth


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_matches_torch_adamw_float64(wd):
    n = 257
    W0 = synth.normal(0, 1, (n,)).astype(np.float64)
    lr, b1, b2, eps = 3e-4, 0.9, 0.95, 1e-8
    p = torch.nn.Parameter(torch.tensor(W0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    W, m, v = W0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 6):
        G = synth.normal(0, 10 + t, (n,)).astype(np.float64) * 1e-3
        p.grad = torch.tensor(G, dtype=torch.float64)
        opt.step()
        W, m, v = oracle.adamw_step(W, G, m, v, lr, b1, b2, eps, wd, t)
        st = opt.state[p]
        np.testing.assert_allclose(W, p.detach().numpy(), rtol=1e-13, atol=1e-16)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-18)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-20)


def test_step_one_closed_form():
    # From zero moments: m_hat = g, v_hat = g^2, so
    # W1 = W0 (1 - lr wd) - lr g / (|g| + eps).
    W0 = synth.normal(1, 1, (64,)).astype(np.float64)
    G = synth.normal(1, 2, (64,)).astype(np.float64)
    lr, wd, eps = 1e-2, 0.1, 1e-8
    W1, _, _ = oracle.adamw_step(W0, G, np.zeros(64), np.zeros(64), lr, 0.9, 0.95, eps, wd, 1)
    np.testing.assert_allclose(W1, W0 * (1 - lr * wd) - lr * G / (np.abs(G) + eps), rtol=1e-13)


def test_zero_grad_zero_state_is_pure_decay():
    W0 = synth.normal(1, 3, (16,)).astype(np.float64)
    W1, m, v = oracle.adamw_step(W0, np.zeros(16), np.zeros(16), np.zeros(16), 1e-3, 0.9, 0.95,
                                 1e-8, 0.1, 1)
    np.testing.assert_array_equal(W1, W0 * (1 - 1e-4))
    assert np.all(m == 0) and np.all(v == 0)
