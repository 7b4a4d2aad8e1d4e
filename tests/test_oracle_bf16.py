"""Pins for the oracle's float64 -> bf16 storage rounding (CPU only)."""
import numpy as np
import torch

import oracle
import synth


def test_matches_torch_on_float32_values():
    # Values exactly representable in float32: torch's bf16 cast is a single
    # round-to-nearest-even, the same rounding the oracle must do.
    x = synth.normal_f32(9, 1, 20000, std=0.02).astype(np.float64)
    want = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), want)


def test_ties_and_near_ties_from_float64():
    one_ulp = 2.0 ** -7
    cases = {
        1.0 + one_ulp / 2: 1.0,                 # tie, even stays
        1.0 + 3 * one_ulp / 2: 1.0 + 2 * one_ulp,  # tie, odd rounds up
        1.0 + one_ulp / 2 + 2 ** -40: 1.0 + one_ulp,  # just above the tie
        1.0 + one_ulp / 2 - 2 ** -40: 1.0,      # just below the tie
        -(1.0 + one_ulp / 2 + 2 ** -40): -(1.0 + one_ulp),
    }
    for x, want in cases.items():
        assert oracle.round_bf16(np.array([x]))[0] == want, x


def test_noncontiguous_input():
    x = synth.normal_f32(9, 2, 64).astype(np.float64).reshape(8, 8)
    np.testing.assert_array_equal(oracle.round_bf16(x.T), oracle.round_bf16(x).T)
