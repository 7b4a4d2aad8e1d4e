"""The seeded input generator (CPU side): definition, determinism, statistics."""
import numpy as np
import torch

import synth


def _scalar_reference(seed, tid, i):
    key = synth.tensor_key(seed, tid)
    s = 0
    for k in range(6):
        w = synth.splitmix64_int((key + 6 * i + k) & ((1 << 64) - 1))
        s += (w & 0xFFFFFFFF) + (w >> 32)
    return np.float32((s - 6 * 2 ** 32) * 2.0 ** -32)


def test_splitmix64_known_values():
    # SplitMix64 from state 0 (first output of the published generator with
    # seed 0) and from state 1 increments.
    assert synth.splitmix64_int(0) == 0xE220A8397B1DCDAF
    assert synth.splitmix64_int(0x9E3779B97F4A7C15) == 0x6E789E6AA1B965F4


def test_vector_matches_scalar_definition():
    got = synth.normal_f32(3, 17, 40, offset=1000)
    want = np.array([_scalar_reference(3, 17, 1000 + i) for i in range(40)], dtype=np.float32)
    np.testing.assert_array_equal(got, want)


def test_offsets_and_chunks_are_consistent():
    full = synth.normal_f32(1, 2, synth.CHUNK + 100)
    part = synth.normal_f32(1, 2, 150, offset=synth.CHUNK - 50)
    np.testing.assert_array_equal(full[synth.CHUNK - 50:], part)


def test_moments_and_support():
    x = synth.normal_f32(0, 0, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert np.abs(x).max() <= 6.0
    assert len(np.unique(synth.normal_f32(0, 1, 1000))) > 990


def test_bf16_rounding_matches_torch():
    x = np.concatenate([synth.normal_f32(0, 5, 10000, std=3.0),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0,
                                  np.inf, -np.inf, 3.3e38, 1e-40], dtype=np.float32)])
    want = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(x), want)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(want),
                                  torch.tensor(x).to(torch.bfloat16).float().numpy())
