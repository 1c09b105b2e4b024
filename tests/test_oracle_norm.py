"""Pins of the oracle's RMSNorm prologue (RMSNorm fused into the activation quantizer) to
facts that do not come from the oracle itself.

- r = 1 / sqrt(mean(x^2) + eps) on rows with closed forms: constant rows with
  eps = 3 c^2 give r = 1 / (2 |c|) exactly; two-level rows against Python's own sqrt;
- gamma acts element by element on the quantized value and not on r: doubling gamma on one
  block doubles exactly that block's scale and leaves every code, every other scale and r
  unchanged; gamma zero on odd columns gives the plain quantizer's codes of x with those
  columns zeroed (the plain quantizer is pinned in test_oracle_pins.py);
- gamma = 1: codes and scales of u are the plain quantizer's codes and scales of x;
- the normalised layer agrees with a dense binary64 textbook evaluation (normalise, then
  multiply by the dequantized weights) within the activation-quantization error bound.
"""
import math

import numpy as np
import pytest

import workloads
from oracle import oracle as O

QK = 32


def _rows(vals, K):
    return np.array([[v] * K for v in vals], np.float32)


def test_constant_rows_closed_form():
    K = 96
    cs = [1.0, -0.75, 2.0 ** -10, 48.0, -3.0 * 2.0 ** 20]
    x = _rows(cs, K)
    for c in cs:
        row = _rows([c], K)
        xq, xd, r = O.rmsnorm_quantize_act(row, np.ones(K, np.float32), eps=3.0 * c * c)
        assert r[0] == 1.0 / (2.0 * abs(c))          # mean = c^2, sqrt(4 c^2) = 2 |c|
        assert np.all(xq == (127 if c > 0 else -127))
        assert np.all(xd == np.float32(abs(c) / 127.0))
    # the same rows in one call: rows are independent
    _, _, r = O.rmsnorm_quantize_act(x, np.ones(K, np.float32), eps=1.0)
    for m, c in enumerate(cs):
        assert r[m] == pytest.approx(1.0 / math.sqrt(c * c + 1.0), rel=1e-15)


@pytest.mark.parametrize("a,b,eps", [(1.0, 3.0, 1e-6), (0.5, -0.25, 0.0625), (100.0, 0.0, 1e-5)])
def test_two_level_rows(a, b, eps):
    K = 128
    x = np.array([[a] * (K // 2) + [b] * (K // 2)], np.float32)
    _, _, r = O.rmsnorm_quantize_act(x, np.ones(K, np.float32), eps)
    want = 1.0 / math.sqrt((float(np.float32(a)) ** 2 + float(np.float32(b)) ** 2) / 2.0 + eps)
    assert r[0] == pytest.approx(want, rel=2e-16)


def test_bf16_rows_use_the_widened_values():
    K = 64
    bits = np.full((1, K), 0x3FC0, np.uint16)  # bf16 1.5
    _, xd, r = O.rmsnorm_quantize_act(bits, np.ones(K, np.float32), eps=3 * 2.25, bf16=True)
    assert r[0] == 1.0 / 3.0 and np.all(xd == np.float32(1.5 / 127))


def test_unit_gamma_gives_the_plain_quantizer():
    rng = np.random.default_rng(1)
    x, _ = workloads.activations(rng, 5, 256, bf16=True, outlier_frac=0.02)
    xq, xd, _ = O.rmsnorm_quantize_act(x, np.ones(256, np.float32), 1e-6, bf16=True)
    xq0, xd0 = O.quantize_act(x, bf16=True)
    assert np.array_equal(xq, xq0) and np.array_equal(xd.view(np.uint32), xd0.view(np.uint32))


def test_gamma_on_one_block_scales_only_that_block():
    rng = np.random.default_rng(2)
    M, K, j = 3, 256, 5
    x = rng.standard_normal((M, K)).astype(np.float32)
    g1 = np.ones(K, np.float32)
    g2 = g1.copy()
    g2[QK * j:QK * (j + 1)] = 2.0
    q1, d1, r1 = O.rmsnorm_quantize_act(x, g1, 1e-6)
    q2, d2, r2 = O.rmsnorm_quantize_act(x, g2, 1e-6)
    assert np.array_equal(q1, q2)
    assert np.array_equal(r1, r2)                       # r comes from x, not from x * gamma
    assert np.array_equal(d2[:, j], 2 * d1[:, j])
    other = [b for b in range(K // QK) if b != j]
    assert np.array_equal(d2[:, other], d1[:, other])


def test_gamma_zero_on_odd_columns():
    rng = np.random.default_rng(3)
    M, K = 4, 128
    x = rng.standard_normal((M, K)).astype(np.float32)
    g = np.ones(K, np.float32)
    g[1::2] = 0.0
    xq, xd, _ = O.rmsnorm_quantize_act(x, g, 1e-6)
    xz = x.copy()
    xz[:, 1::2] = 0.0
    xq0, xd0 = O.quantize_act(xz)
    assert np.array_equal(xq, xq0) and np.array_equal(xd, xd0)
    assert not np.any(xq[:, 1::2])


@pytest.mark.parametrize("M,N,K,bf16", [(5, 7, 96, False), (9, 40, 512, True)])
def test_normalised_layer_within_the_quantization_bound(M, N, K, bf16):
    rng = np.random.default_rng(M * 100 + N)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=bf16, outlier_frac=0.02)
    x32 = workloads.f32_from_bf16_bits(x) if bf16 else x
    gamma = (0.5 + rng.random(K)).astype(np.float32)
    eps = 1e-5
    Wq, Wd = O.quantize_weights(W)
    xq, xd, r = O.rmsnorm_quantize_act(x, gamma, eps, bf16=bf16)
    y = O.linear_epilogue(xq, xd, Wq, Wd, rowscale=r).astype(np.float64)
    # textbook: normalise in binary64, then multiply by the dequantized weights
    X = x32.astype(np.float64)
    rt = 1.0 / np.sqrt(np.mean(X * X, axis=1) + eps)
    Z = X * rt[:, None] * gamma.astype(np.float64)[None, :]
    Wdq = Wq.astype(np.float64) * np.repeat(Wd.view(np.float16).astype(np.float64), QK, axis=1)
    dense = Z @ Wdq.T
    # activation error per element: half a code step of the normalised scale, plus the
    # binary32 rounding of x * gamma, both carried by r
    step = np.repeat(xd.astype(np.float64), QK, axis=1) * rt[:, None]
    ez = step * (0.5 + 1e-6) + np.abs(Z) * 2.0 ** -23
    bound = ez @ np.abs(Wdq).T + 2.0 ** -23 * np.abs(dense) + 1e-30
    assert np.all(np.abs(y - dense) <= bound)
    assert np.max(np.abs(y - dense)) > 0
