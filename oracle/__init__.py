"""Plain fp64 CPU oracle of the hybrid Muon + AdamW optimizer step.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package. The CUDA library and its Python
binding never do, and the two share no code: the only common dependency is
the seeded input generator in ``synth``.

Parity pins (each in tests/test_oracle_*.py) tie every function here to
something other than itself: closed forms, the SVD of the input, invariances
the iteration must respect, brute force on tiny inputs, and PyTorch's own
AdamW and gradient clipping in float64.
"""
from .muon import (NS_COEFFS, NS_EPS, NS_STEPS, NORMUON_FLOOR, CAUTIOUS_OFF, CAUTIOUS_UPDATE,
                   CAUTIOUS_WD, SHAPE_MOONLIGHT, SHAPE_RATIO,
                   MuonHparams, momentum_nesterov, muon_apply, muon_plus_row_col,
                   muon_step_tensor, muon_step_view, newton_schulz, normuon, shape_scale)
from .adamw import adamw_step
from .bf16 import round_bf16
from .ns_bf16 import newton_schulz_stored, round_to_bits
from .grad_control import CLIP_EPS, GradControl, grad_control
from .qk_clip import ClipEntry, gamma, qk_clip
from .stochastic_round import (MOMENT_FIRST, MOMENT_PARAM, MOMENT_SECOND, round_bf16_with_noise,
                               fmix32, sr_key, sr_noise16, sr_stream, stochastic_round_bf16)

__all__ = [
    "NS_COEFFS", "NS_EPS", "NS_STEPS", "NORMUON_FLOOR", "CAUTIOUS_OFF", "CAUTIOUS_UPDATE",
    "CAUTIOUS_WD", "SHAPE_MOONLIGHT", "SHAPE_RATIO",
    "MuonHparams", "momentum_nesterov", "muon_apply", "muon_plus_row_col", "muon_step_tensor",
    "muon_step_view", "newton_schulz", "newton_schulz_stored", "normuon", "round_to_bits",
    "shape_scale", "adamw_step", "round_bf16",
    "CLIP_EPS", "GradControl", "grad_control", "MOMENT_FIRST", "MOMENT_PARAM", "MOMENT_SECOND",
    "round_bf16_with_noise", "fmix32", "sr_key", "sr_noise16", "sr_stream",
    "stochastic_round_bf16", "ClipEntry", "gamma", "qk_clip",
]
