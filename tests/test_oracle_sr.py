"""Pins of the stochastic-rounding oracle (dew.training.optim,
"stochastic_round_bf16" and "bf16_moments")."""
import numpy as np
import pytest

import oracle


def _bits(x32):
    return np.asarray(x32, dtype=np.float32).view(np.uint32)


def test_fmix32_published_values():
    """MurmurHash3_x86_32 of the empty input is fmix32(seed): the published
    test vectors for seeds 0, 1 and 0xFFFFFFFF."""
    assert oracle.fmix32(0) == 0
    assert oracle.fmix32(1) == 0x514E28B7
    assert oracle.fmix32(0xFFFFFFFF) == 0x81F16F39
    vec = oracle.fmix32(np.array([0, 1, 0xFFFFFFFF], dtype=np.uint64))
    assert list(map(int, vec)) == [0, 0x514E28B7, 0x81F16F39]


@pytest.mark.parametrize("pattern", [0x3F800001, 0x3F807FFF, 0x3F808000, 0x3F80FFFF, 0xBF812345,
                                     0x00012345, 0x7F7F0001])
def test_round_up_probability_is_the_dropped_fraction(pattern):
    """Over all 65536 noise values the result rounds up exactly `dropped`
    times, and it is always one of the two bf16 neighbours."""
    x = np.array([pattern], dtype=np.uint32).view(np.float32).astype(np.float64)
    noise = np.arange(65536, dtype=np.uint32)
    out = oracle.round_bf16_with_noise(np.repeat(x, 65536), noise)
    down = np.array([pattern & 0xFFFF0000], dtype=np.uint32).view(np.float32)[0]
    up = np.array([(pattern & 0xFFFF0000) + 0x10000], dtype=np.uint32).view(np.float32)[0]
    n_up = int(np.sum(out == np.float64(up)))
    assert n_up + int(np.sum(out == np.float64(down))) == 65536
    assert n_up == pattern & 0xFFFF


def test_representable_values_never_move():
    vals = np.array([1.0, -2.5, 0.0, 3.0e38, 1.0e-40, -7.8125e-3], dtype=np.float32)
    vals = (_bits(vals) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    for r in (0, 1, 0x7FFF, 0xFFFF):
        np.testing.assert_array_equal(oracle.round_bf16_with_noise(vals, np.full(vals.shape, r)),
                                      vals)


def test_nan_inf_and_signed_zero():
    low_payload_nan = np.array([0x7F800001, 0xFF800001], dtype=np.uint32).view(np.float32)
    for r in (0, 0xFFFF):
        out = oracle.round_bf16_with_noise(low_payload_nan, [r, r])
        assert np.all(np.isnan(out))
        assert np.signbit(out[1]) and not np.signbit(out[0])
    out = oracle.round_bf16_with_noise(np.array([np.inf, -np.inf, -0.0]), [0xFFFF] * 3)
    assert out[0] == np.inf and out[1] == -np.inf and out[2] == 0.0 and np.signbit(out[2])


def test_largest_finite_rounds_to_inf_with_its_dropped_fraction():
    x = np.array([0x7F7FFFFF], dtype=np.uint32).view(np.float32).astype(np.float64)
    out = oracle.round_bf16_with_noise(np.repeat(x, 65536), np.arange(65536))
    assert int(np.sum(np.isinf(out))) == 0xFFFF


def test_unbiased_in_expectation():
    x = 1.0 + 0.3 * 2.0 ** -7             # 30 % of the way to the next bf16 value
    n = 1 << 20
    out = oracle.stochastic_round_bf16(np.full(n, x), seed=11, stream=oracle.sr_stream(3, 0))
    ulp = 2.0 ** -7
    p = 0.3
    sigma = ulp * np.sqrt(p * (1 - p) / n)
    assert abs(out.mean() - np.float64(np.float32(x))) < 5 * sigma
    assert set(np.unique(out)) == {1.0, 1.0 + ulp}


def test_noise_is_uniform_and_streams_differ():
    idx = np.arange(1 << 18, dtype=np.uint64)
    a = oracle.sr_noise16(oracle.sr_key(5, oracle.sr_stream(0, 0)), idx).astype(np.int64)
    b = oracle.sr_noise16(oracle.sr_key(5, oracle.sr_stream(0, 1)), idx).astype(np.int64)
    c = oracle.sr_noise16(oracle.sr_key(6, oracle.sr_stream(0, 0)), idx).astype(np.int64)
    hist = np.bincount(a >> 12, minlength=16)          # 16 bins of 4096 values
    expect = len(idx) / 16
    chi2 = float(np.sum((hist - expect) ** 2 / expect))
    assert chi2 < 45.0                                  # 15 dof: p ~ 1e-4
    for other in (b, c):
        assert abs(np.corrcoef(a, other)[0, 1]) < 0.02
    # a pure function of (seed, stream, index)
    np.testing.assert_array_equal(
        a, oracle.sr_noise16(oracle.sr_key(5, oracle.sr_stream(0, 0)), idx).astype(np.int64))


def test_one_hash_serves_two_elements():
    key = oracle.sr_key(3, oracle.sr_stream(1, 2))
    h = oracle.fmix32((key + 10) & 0xFFFFFFFF)
    got = oracle.sr_noise16(key, np.arange(20, 22, dtype=np.uint64))
    assert list(map(int, got)) == [h & 0xFFFF, h >> 16]


def test_key_uses_both_halves_of_the_seed():
    s = oracle.sr_stream(0, 0)
    assert oracle.sr_key(5, s) != oracle.sr_key(5 + (1 << 32), s)
    assert oracle.sr_key(5, s) != oracle.sr_key(5, oracle.sr_stream(0, 1))


def test_small_increments_survive_in_expectation():
    """dew "bf16_moments": at b2 = 0.999 round-to-nearest loses every
    increment below half a bf16 spacing, stochastic rounding keeps them in
    expectation. v <- b2 v + (1-b2) * 2 from v = 1: fp64 reaches 2 - 0.999^t."""
    b2, steps, n = 0.999, 1000, 512
    v_sr = np.ones(n)
    v_rn = np.ones(n)
    for t in range(steps):
        v_sr = oracle.stochastic_round_bf16(b2 * v_sr + (1 - b2) * 2.0, seed=t + 1,
                                            stream=oracle.sr_stream(0, oracle.MOMENT_SECOND))
        v_rn = oracle.round_bf16(b2 * v_rn + (1 - b2) * 2.0)
    exact = 2.0 - b2 ** steps
    assert np.all(v_rn == 1.0)                       # nearest rounding never moves
    assert abs(v_sr.mean() - exact) < 0.01           # SR follows fp64 in expectation
