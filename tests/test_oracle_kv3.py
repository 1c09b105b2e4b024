"""Pins of the 3-bit KV-cache codec oracle (oracle/kv3_oracle.c) to facts that do not come
from the oracle itself.

- the transform: scipy's Sylvester Hadamard matrix on integer vectors (exact), and the
  transform applied twice is 128 times the identity;
- the codebook: Max's (1960) 8-level table for the unit Gaussian satisfies the Lloyd-Max
  conditions (each level the conditional mean of its cell, each threshold the midpoint of
  its neighbours), and its distortion is the tabulated 0.03454;
- the decoder's levels: a group of equal codes decodes to (+-level, 0, ..., 0);
- the decision thresholds: a probe element p among 127 unit values flips its code at the
  closed-form point |p| = t * sqrt(127 / (128 - t^2)) (where |p| = t * RMS);
- the bit layout and signs: a scaled unit vector rotates to +-c times a Hadamard column,
  so its codes are 1 or 5 following that column's signs, and it decodes to 0.7560 c e_j
  exactly;
- the scale is the RMS of the rotated group (binary64 reference, a few ulp);
- the rotation spreads outlier channels: the distortion stays the Gaussian one.
"""
import math

import numpy as np
import pytest

from oracle import kv3

scipy_linalg = pytest.importorskip("scipy.linalg")
scipy_stats = pytest.importorskip("scipy.stats")
H = scipy_linalg.hadamard(128).astype(np.float64)
TABLE_LEVELS = (0.2451, 0.7560, 1.3440, 2.1520)   # Max (1960), N = 8, unit Gaussian
TABLE_THRESHOLDS = (0.5006, 1.0500, 1.7480)
TABLE_MSE = 0.03454


def test_fwht_is_the_sylvester_hadamard_matrix():
    rng = np.random.default_rng(0)
    for _ in range(20):
        x = rng.integers(-1000, 1000, 128).astype(np.float32)
        assert np.array_equal(kv3.fwht(x).astype(np.float64), H @ x.astype(np.float64))
    e = np.zeros(128, np.float32)
    e[37] = 1.0
    assert np.array_equal(kv3.fwht(e), H[:, 37].astype(np.float32))


def test_fwht_twice_is_128_times_identity():
    x = np.random.default_rng(1).integers(-50, 50, 128).astype(np.float32)
    assert np.array_equal(kv3.fwht(kv3.fwht(x)), 128 * x)


def test_max_table_satisfies_the_lloyd_max_conditions():
    norm = scipy_stats.norm
    edges = (0.0,) + TABLE_THRESHOLDS + (math.inf,)
    for k, level in enumerate(TABLE_LEVELS):
        a, b = edges[k], edges[k + 1]
        centroid = (norm.pdf(a) - norm.pdf(b)) / (norm.cdf(b) - norm.cdf(a))
        assert centroid == pytest.approx(level, abs=1.5e-3)
    for k, t in enumerate(TABLE_THRESHOLDS):
        assert t == pytest.approx((TABLE_LEVELS[k] + TABLE_LEVELS[k + 1]) / 2, abs=1e-4)
    mse = 0.0
    for k, level in enumerate(TABLE_LEVELS):
        a, b = edges[k], edges[k + 1]
        # E[(X - level)^2 ; a < X < b] for the unit Gaussian, both signs
        m0 = norm.cdf(b) - norm.cdf(a)
        m1 = norm.pdf(a) - norm.pdf(b)
        m2 = m0 + (a * norm.pdf(a) if a > 0 else 0.0) - (b * norm.pdf(b) if math.isfinite(b) else 0.0)
        mse += 2 * (m2 - 2 * level * m1 + level * level * m0)
    assert mse == pytest.approx(TABLE_MSE, abs=2e-4)


def _words_all(code):
    """12 words holding 128 copies of one 3-bit code (written bit by bit)."""
    bits = np.zeros(384, np.uint8)
    for i in range(128):
        for j in range(3):
            bits[3 * i + j] = (code >> j) & 1
    return np.packbits(bits, bitorder="little").view(np.uint32).reshape(1, 12)


@pytest.mark.parametrize("code", range(8))
def test_decoder_levels_are_the_table(code):
    out = kv3.decode(_words_all(code), np.array([1.0], np.float32))[0]
    level = TABLE_LEVELS[code & 3] * (-1 if code & 4 else 1)
    assert out[0] == np.float32(level)
    assert not np.any(out[1:])


@pytest.mark.parametrize("k", range(3))
def test_decision_thresholds_from_the_closed_form(k):
    t = TABLE_THRESHOLDS[k]
    p_star = t * math.sqrt(127.0 / (128.0 - t * t))   # |p| = t * RMS of (p, 1, ..., 1)
    for sign in (1.0, -1.0):
        for rel, want in ((1 - 1e-4, k), (1 + 1e-4, k + 1)):
            u = np.ones(128)
            u[5] = sign * p_star * rel
            x = (H @ u / 128.0).astype(np.float32)      # rotates back to u (to rounding)
            words, _ = kv3.encode(x[None, :])
            c = kv3.codes(words)[0]
            assert c[5] == want + (4 if sign < 0 else 0), (k, sign, rel, c[5])
            assert np.all(c[np.arange(128) != 5] == 1)   # |1| / RMS is about 1: cell 1


@pytest.mark.parametrize("j,c", [(0, 1.0), (37, -0.5), (127, 8.0), (64, -2.0 ** -20)])
def test_unit_vector_codes_layout_and_exact_round_trip(j, c):
    x = np.zeros((1, 128), np.float32)
    x[0, j] = c
    words, scales = kv3.encode(x)
    assert scales[0] == abs(c)                           # sqrt(128 c^2 / 128)
    want = np.where(c * H[:, j] < 0, 5, 1)               # cell 1, sign of the column
    assert np.array_equal(kv3.codes(words)[0], want)
    y = kv3.decode(words, scales)[0]
    expect = np.zeros(128, np.float32)
    expect[j] = np.float32(0.7560) * np.float32(c)
    assert np.array_equal(y, expect)


def test_zero_group():
    words, scales = kv3.encode(np.zeros((3, 128), np.float32))
    assert not np.any(words) and not np.any(scales)
    assert not np.any(kv3.decode(words, scales))


def test_scale_is_the_rms_of_the_rotated_group():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((200, 128)).astype(np.float32) * 10.0 ** rng.integers(-3, 4, (200, 1))
    _, scales = kv3.encode(x)
    ref = np.sqrt(np.mean((x.astype(np.float64) @ H.T) ** 2, axis=1))
    assert np.all(np.abs(scales - ref) <= 8 * np.spacing(ref.astype(np.float32)))


def test_bf16_groups_use_the_widened_values():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 128)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)           # truncate to bf16
    x16 = (bits.astype(np.uint32) << 16).view(np.float32)
    a = kv3.encode(bits, bf16=True)
    b = kv3.encode(x16)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gaussian_distortion_is_the_lloyd_max_one():
    x = np.random.default_rng(4).standard_normal((4000, 128)).astype(np.float32)
    y = kv3.decode(*kv3.encode(x))
    rel = np.sum((x - y) ** 2) / np.sum(x ** 2)
    assert rel == pytest.approx(TABLE_MSE, abs=0.004)


def test_rotation_spreads_outlier_channels():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4000, 128)).astype(np.float32)
    x[:, [3, 70, 101]] *= 30.0                        # three outlier channels
    y = kv3.decode(*kv3.encode(x))
    rel = np.sum((x - y) ** 2) / np.sum(x ** 2)
    assert rel < 0.045
    # without the rotation (codes of x itself on its RMS scale) the same data does worse
    s = np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True))
    z = np.abs(x / s)
    cells = np.searchsorted(TABLE_THRESHOLDS, z, side="right")
    q = np.sign(x) * np.asarray(TABLE_LEVELS)[cells] * s
    assert np.sum((x - q) ** 2) / np.sum(x ** 2) > 1.5 * rel


def test_exact_zeros_get_the_positive_code():
    """x = e_0 + e_1 rotates to H[:,0] + H[:,1]: 64 exact zeros and 64 twos, RMS sqrt(2).
    |2| / sqrt(2) = 1.414 lies in cell 2; a zero is cell 0 with the positive sign (u < 0 is
    false)."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = x[0, 1] = 1.0
    words, scales = kv3.encode(x)
    u = H[:, 0] + H[:, 1]
    assert scales[0] == np.float32(math.sqrt(2.0))
    assert np.array_equal(kv3.codes(words)[0], np.where(u == 0, 0, 2))


def test_negative_zero_rotation_output_gets_the_positive_code():
    """x = -0 e_0 + 5 e_2 + 5 e_3.  The last output of the rotation is
    ((-0 - 0) - (5 - 5)) - 0 - ... (it takes the difference at every stage, and every later
    subtrahend is an exact +0); IEEE subtraction gives -0 - (+0) = -0, so it is a negative
    zero while the group's RMS is not 0.  u < 0 is false for it,
    so its code is 0 (cell 0, positive sign), like a +0."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = -0.0
    x[0, 2] = x[0, 3] = 5.0
    u = np.asarray(kv3.fwht(x[0]), np.float32)
    assert u[127] == 0 and np.signbit(u[127])
    words, scales = kv3.encode(x)
    assert scales[0] == np.sqrt(np.float32(50.0))  # 64 outputs of +-10: ss / 128 = 50
    assert kv3.codes(words)[0][127] == 0
