"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one part of the oracle to the Q8_0 definition, to hand-worked values
(tests/golden), to a library routine for a special case (numpy's binary16 conversion),
to brute force on tiny inputs, or to the quantization error bound against the dense
binary64 product.  A dropped term, a wrong sign or index, a transposed operand or a
wrong rounding mode in the oracle fails at least one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import oracle as O
from tests import brute_q8 as B

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
QK = 32


def _block_from(nz):
    v = np.zeros(QK, np.float32)
    for k, val in nz.items():
        v[int(k)] = val
    return v


# --------------------------------------------------------------------------- #
# binary16 conversion: a special case that reduces to a library routine       #
# --------------------------------------------------------------------------- #

def test_f32_to_f16_matches_numpy_rne():
    rng = np.random.default_rng(123)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -14, 2.0 ** -24,
            2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -25, 2.0 ** -26, 1e-30, 5.960464477539063e-08,
            6.097555160522461e-05, 0.1, 1 / 3, 2047.0, 2049.0, 2051.0, 4095.0, 4097.0]
    # exact midpoints between binary16 neighbours at several exponents (ties to even)
    for e in range(-24, 16):
        for m in (0, 1, 2, 3, 1021, 1022, 1023):
            base = (1024 + m) * 2.0 ** (e - 10) if e >= -14 else m * 2.0 ** -24
            vals.append(base + 2.0 ** (max(e, -14) - 11))
    vals += list(rng.standard_normal(20000).astype(np.float32) * 0.001)
    vals += list((rng.random(20000) * 1e-4).astype(np.float32))
    vals += list(np.exp(rng.uniform(-20, 11, 20000)).astype(np.float32))
    arr = np.array(vals, dtype=np.float32)
    arr = np.concatenate([arr, -arr])
    with np.errstate(over="ignore"):
        want = arr.astype(np.float16).view(np.uint16)
    got = np.array([O.f32_to_f16_bits(float(v)) for v in arr], dtype=np.uint16)
    bad = np.nonzero(want != got)[0]
    assert bad.size == 0, [(float(arr[i]), hex(want[i]), hex(got[i])) for i in bad[:10]]


def test_f16_to_f64_all_finite_codes():
    bits = np.arange(0, 0x10000, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    got = np.array([O.f16_bits_to_f64(int(b)) for b in bits[fin]])
    assert np.array_equal(got, ref[fin])


# --------------------------------------------------------------------------- #
# P4: hand-worked blocks (ties, exact scales, zero block)                       #
# --------------------------------------------------------------------------- #

def test_golden_tie_blocks():
    g = json.load(open(os.path.join(GOLDEN, "q8_0_ties.json")))
    for case in g["cases"]:
        v = _block_from(case["block_nonzero"])
        q, d = O.quantize_block(v)
        want = np.zeros(QK, np.int8)
        for k, c in case["codes_nonzero"].items():
            want[int(k)] = c
        assert np.array_equal(q, want), case["name"]
        assert float(d) == case["d32"], case["name"]
        if case["d16_bits"] is not None:
            assert O.f32_to_f16_bits(float(d)) == case["d16_bits"], case["name"]
        else:
            case["d16_bits"] = int(np.float32(case["d32"]).astype(np.float16).view(np.uint16))
        # where the fixture states exact ratios, check them with rational arithmetic
        ex = case.get("exact")
        if ex:
            dd = Fraction(case["d32"])
            amax = max(abs(Fraction(float(val))) for val in case["block_nonzero"].values())
            assert amax == ex["amax_over_d"] * dd
            for k, ratio in ex["w_over_d"].items():
                assert Fraction(float(case["block_nonzero"][k])) == Fraction(ratio) * dd
        # the same block as weights: codes + binary16 scale
        Wq, Wd = O.quantize_weights(v[None, :])
        assert np.array_equal(Wq[0], want) and int(Wd[0, 0]) == case["d16_bits"]
        # half-to-even rounding would differ exactly where the fixture says
        for k, c in case.get("half_even_would_give", {}).items():
            assert int(q[int(k)]) != c


# --------------------------------------------------------------------------- #
# P1-P3, P5: invariants of the block quantizer                                  #
# --------------------------------------------------------------------------- #

def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    blocks = rng.standard_normal((n, QK)).astype(np.float32)
    scales = np.exp(rng.uniform(-30, 30, size=(n, 1))).astype(np.float32)
    blocks = (blocks * scales).astype(np.float32)
    # a few blocks with exact ties, repeated amax, single nonzero, constant values
    blocks[0] = np.float32(0.5) * np.arange(-16, 16, dtype=np.float32)
    blocks[1] = np.float32(-3.0)
    blocks[2] = 0.0
    blocks[2, 7] = np.float32(1e-3)
    blocks[3] = np.where(np.arange(QK) % 2 == 0, 127.0, -127.0).astype(np.float32)
    return blocks


def test_roundtrip_bound_and_extreme_codes():
    blocks = _random_blocks(4000, 1)
    Xq, Xd = O.quantize_act(blocks.reshape(1, -1))
    Xq = Xq.reshape(-1, QK).astype(np.float64)
    Xd = Xd.reshape(-1).astype(np.float64)
    W = blocks.astype(np.float64)
    for i in range(blocks.shape[0]):
        d = Xd[i]
        amax = np.max(np.abs(W[i]))
        assert d == np.float64(np.float32(np.float32(amax) / np.float32(127.0)))
        err = np.abs(W[i] - Xq[i] * d)
        # P1: |w - q d| <= d (1/2 + 128 * 2^-24)   (binary32 rounding of w/d included)
        assert np.all(err <= d * (0.5 + 128 * 2.0 ** -24)), i
        # P3: the amax element gets |q| = 127; signs agree; |q| <= 127
        j = int(np.argmax(np.abs(W[i])))
        assert abs(Xq[i, j]) == 127
        assert np.all(np.abs(Xq[i]) <= 127)
        assert np.all((Xq[i] == 0) | (np.sign(Xq[i]) == np.sign(W[i])))


def test_roundtrip_bound_with_binary16_weight_scale():
    W = workloads.weights(np.random.default_rng(5), 64, 512)
    Wq, Wd = O.quantize_weights(W)
    d16 = Wd.view(np.float16).astype(np.float64)
    W64 = W.astype(np.float64).reshape(64, -1, QK)
    q = Wq.astype(np.float64).reshape(64, -1, QK)
    amax = np.abs(W64).max(axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    err = np.abs(W64 - q * d16[:, :, None])
    bound = d32 * (0.5 + 128 * 2.0 ** -24) + 127 * np.abs(d32 - d16)
    assert np.all(err <= bound[:, :, None])
    # the stored scale is the binary16 rounding of amax/127
    assert np.array_equal(Wd, d32.astype(np.float32).astype(np.float16).view(np.uint16))


def test_all_zero_block_gives_zero_scale_and_codes():
    x = np.zeros((3, 96), np.float32)
    x[1, 32:64] = -0.0
    x[2, 70] = 1.0  # only the third block of row 2 is nonzero
    xq, xd = O.quantize_act(x)
    assert np.all(xq[:2] == 0) and np.all(xd[:2] == 0)
    assert np.all(xd[2, :2] == 0) and xd[2, 2] == np.float32(1.0) / np.float32(127.0)
    Wq, Wd = O.quantize_weights(x)
    assert np.all(Wd[:2] == 0) and np.all(Wd[2, :2] == 0)
    assert Wq[2, 70] == 127 and np.count_nonzero(Wq) == 1


def test_scale_invariance_power_of_two():
    blocks = _random_blocks(500, 2)
    blocks = blocks / np.abs(blocks).max(axis=1, keepdims=True).clip(min=1e-30)
    blocks = blocks.astype(np.float32)
    blocks[2] = 0.0
    for k in (-20, -7, -1, 1, 5, 20):
        s = np.float32(2.0 ** k)
        q0, d0 = O.quantize_act(blocks.reshape(1, -1))
        q1, d1 = O.quantize_act((blocks * s).reshape(1, -1))
        assert np.array_equal(q0, q1)
        assert np.array_equal(d1, (d0 * s).astype(np.float32))


def test_bf16_path_equals_widened_f32_path():
    xb, _ = workloads.activations(np.random.default_rng(9), 7, 256, bf16=True,
                                  outlier_frac=0.05)
    q1, d1 = O.quantize_act(xb, bf16=True)
    q2, d2 = O.quantize_act(workloads.f32_from_bf16_bits(xb))
    assert np.array_equal(q1, q2) and np.array_equal(d1, d2)


def test_subnormal_scale_codes_stay_in_range():
    # amax in the binary32 subnormal range: d32 carries few bits, the clamp keeps |q|<=127
    v = np.zeros((1, 64), np.float32)
    v[0, :32] = np.float32(3e-43) * np.linspace(-1, 1, 32, dtype=np.float32)
    v[0, 32] = np.float32(1e-45)  # d32 underflows to 0: codes 0, scale 0
    q, d = O.quantize_act(v)
    assert np.all(np.abs(q.astype(int)) <= 127)
    assert d[0, 1] == 0 and np.all(q[0, 32:] == 0)


# --------------------------------------------------------------------------- #
# P6: block sums against brute force in Python integers                        #
# --------------------------------------------------------------------------- #

def test_block_sums_brute_force():
    rng = np.random.default_rng(11)
    for M, N, K in ((1, 1, 32), (3, 4, 64), (4, 2, 96)):
        xq = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
        wq = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        got = O.block_sums(xq, wq)
        for m in range(M):
            for n in range(N):
                for b in range(K // QK):
                    s = sum(int(xq[m, b * QK + j]) * int(wq[n, b * QK + j]) for j in range(QK))
                    assert got[m, n, b] == s
    ones = np.full((2, 64), 127, np.int8)
    ones[1] = -127
    got = O.block_sums(ones, ones)
    assert got[0, 0, 0] == 516128 and got[0, 1, 1] == -516128 and got[1, 1, 0] == 516128


# --------------------------------------------------------------------------- #
# P8: closed form with unit codes and hand-picked scales                       #
# --------------------------------------------------------------------------- #

def test_closed_form_unit_codes():
    g = json.load(open(os.path.join(GOLDEN, "q8_0_closed_form.json")))
    M, N, K = g["M"], g["N"], g["K"]
    xq = np.ones((M, K), np.int8)
    wq = np.ones((N, K), np.int8)
    xd = np.array(g["d_x"], np.float32)
    wd = np.array(g["d_w"], np.float32).astype(np.float16).view(np.uint16)
    y = O.linear_codes(xq, xd, wq, wd, nthreads=1)
    assert np.array_equal(y, np.array(g["y"], np.float32))
    # one-hot codes pick single products: row m, column n, block b, position j
    xq = np.zeros((M, K), np.int8)
    wq = np.zeros((N, K), np.int8)
    xq[1, 40] = 5
    wq[2, 40] = -7
    y = O.linear_codes(xq, xd, wq, wd, nthreads=2)
    want = np.zeros((M, N), np.float32)
    want[1, 2] = np.float32(-35 * g["d_x"][1][1] * g["d_w"][2][1])
    assert np.array_equal(y, want)


# --------------------------------------------------------------------------- #
# P7: quantization error bound against the dense binary64 product              #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("M,N,K,bf16", [(5, 7, 96, False), (16, 40, 512, True), (3, 33, 4096, True)])
def test_linear_within_quantization_bound(M, N, K, bf16):
    rng = np.random.default_rng(M * 1000 + N)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=bf16, outlier_frac=0.02)
    x32 = workloads.f32_from_bf16_bits(x) if bf16 else x
    Wq, Wd = O.quantize_weights(W)
    y = O.linear(x, Wq, Wd, bf16=bf16, nthreads=3).astype(np.float64)
    xq, xd = O.quantize_act(x, bf16=bf16)
    X = x32.astype(np.float64)
    Wf = W.astype(np.float64)
    dense = X @ Wf.T
    # per-element dequantization errors: weight uses the binary16 scale it stores
    d16 = np.repeat(Wd.view(np.float16).astype(np.float64), QK, axis=1)
    ew = np.abs(Wf - Wq.astype(np.float64) * d16)
    ex = np.abs(X - xq.astype(np.float64) * np.repeat(xd.astype(np.float64), QK, axis=1))
    bound = np.abs(X) @ ew.T + ex @ np.abs(Wf).T + ex @ ew.T
    slack = 1e-6 * (np.abs(X) @ np.abs(Wf).T) + 1e-30
    assert np.all(np.abs(y - dense) <= bound + slack)
    # and the error is really of quantization size, not zero (guards a no-op quantizer)
    assert np.max(np.abs(y - dense)) > 0
    # the dequantized product, computed densely in binary64, agrees to binary32 rounding
    deq = (xq.astype(np.float64) * np.repeat(xd, QK, axis=1)) @ (Wq.astype(np.float64) * d16).T
    assert np.all(np.abs(y - deq) <= 2.0 ** -23 * np.abs(deq) + 1e-30 + 1e-12 * np.abs(
        (np.abs(xq) * np.repeat(xd, QK, axis=1)) @ (np.abs(Wq) * d16).T))


def test_transposed_weights_fail_the_bound():
    # a planted mistake in the oracle's use (W instead of W^T) must be caught by P7's check
    rng = np.random.default_rng(3)
    W = workloads.weights(rng, 64, 64)
    x, _ = workloads.activations(rng, 64, 64, bf16=False)
    Wq, Wd = O.quantize_weights(W)
    y_wrong = O.linear(x, *O.quantize_weights(np.ascontiguousarray(W.T)), nthreads=1)
    dense = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.max(np.abs(y_wrong - dense)) > 10 * np.max(np.abs(O.linear(x, Wq, Wd) - dense))


# --------------------------------------------------------------------------- #
# P9: an independent pure-Python implementation agrees on the tiny workload    #
# --------------------------------------------------------------------------- #

def test_independent_python_brute_force_on_tiny_workload():
    wl = workloads.WORKLOADS["tiny"]
    W = wl.make_weights(0)
    x, _ = wl.make_act(0, 0)
    # keep the pure-Python part to a few seconds: all rows, a slice of output columns
    W = W[:48]
    Wq, Wd = O.quantize_weights(W)
    xq, xd = O.quantize_act(x)
    bwc, bws = B.quant_rows(W)
    bxc, bxs = B.quant_rows(x)
    assert np.array_equal(Wq, np.array(bwc, np.int8))
    assert np.array_equal(Wd, np.array([[B.f16_bits(d) for d in r] for r in bws], np.uint16))
    assert np.array_equal(xq, np.array(bxc, np.int8))
    assert np.array_equal(xd, np.array(bxs, np.float32))
    isum = O.block_sums(xq, Wq)
    for m in (0, 7, 15):
        for n in (0, 13, 47):
            for b in range(x.shape[1] // QK):
                assert isum[m, n, b] == B.block_sum(bxc[m], bwc[n], b)
    y = O.linear_codes(xq, xd, Wq, Wd, nthreads=1)
    yb = B.linear_exact(bxc, bxs, bwc, [[B.f16_bits(d) for d in r] for r in bws])
    # binary64 accumulation then one rounding vs exact rational then one rounding:
    # equal, or one binary32 ulp apart when the exact value sits on a rounding edge
    ulp = np.spacing(np.abs(yb))
    assert np.all(np.abs(y.astype(np.float64) - yb.astype(np.float64)) <= ulp)
    assert np.mean(y == yb) > 0.999


def test_sampled_outputs_equal_full_product():
    rng = np.random.default_rng(4)
    W = workloads.weights(rng, 33, 160)
    x, _ = workloads.activations(rng, 9, 160)
    Wq, Wd = O.quantize_weights(W)
    xq, xd = O.quantize_act(x, bf16=True)
    y = O.linear_codes(xq, xd, Wq, Wd, nthreads=4)
    rows = rng.integers(0, 9, 50)
    cols = rng.integers(0, 33, 50)
    assert np.array_equal(O.linear_codes_at(xq, xd, Wq, Wd, rows, cols), y[rows, cols])
    y1 = O.linear_codes(xq, xd, Wq, Wd, nthreads=1)
    assert np.array_equal(y, y1)
