"""Pins of the oracle's fused epilogue (the layer's neighbours: residual add, SiLU-gated
unit, bfloat16 output) to facts that do not come from the oracle itself.

- bfloat16 rounding: hand-worked ties, subnormals and overflow, and torch's own
  binary32 -> bfloat16 conversion on values that binary32 holds exactly (where rounding
  from binary64 and from binary32 are the same operation);
- SiLU: the closed form silu(ln 3) = (3/4) ln 3 (1 / (1 + 1/3) = 3/4), silu(0) = 0 and
  the limits;
- the epilogue wiring: with zero weights y is aux itself; with no op it is the already
  pinned rescaled block sums; on the unit-code closed form it multiplies by a known gate.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as O

torch = pytest.importorskip("torch")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_rounding_hand_worked():
    cases = {
        1.0: 0x3F80,
        -2.0: 0xC000,
        1 + 2 ** -8: 0x3F80,                 # tie between 1 and 1 + 2^-7: to even (1)
        1 + 3 * 2 ** -8: 0x3F82,             # tie between 1 + 2^-7 and 1 + 2^-6: to even
        1 + 2 ** -8 + 2 ** -30: 0x3F81,      # just above the tie
        1 + 2 ** -8 - 2 ** -30: 0x3F80,      # just below the tie
        2.0 ** -126: 0x0080,                 # smallest normal
        2.0 ** -133: 0x0001,                 # smallest subnormal
        1.5 * 2.0 ** -133: 0x0002,           # subnormal tie: to even
        2.5 * 2.0 ** -133: 0x0002,
        2.0 ** -135: 0x0000,                 # rounds to zero (below half the smallest subnormal)
        (2 - 2 ** -7) * 2.0 ** 127: 0x7F7F,  # largest finite
        (2 - 2 ** -8) * 2.0 ** 127: 0x7F80,  # halfway to 2^128: ties to even -> overflow
        1e39: 0x7F80,
        0.0: 0x0000,
    }
    for v, bits in cases.items():
        assert O.f64_to_bf16(v) == bits, (v, hex(O.f64_to_bf16(v)), hex(bits))
    assert O.f64_to_bf16(-0.0) == 0x8000


def test_bf16_rounding_matches_torch_on_binary32_values():
    rng = np.random.default_rng(5)
    wide = rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)
    bits = rng.integers(0, 0x7F800000, 5000, dtype=np.int64).astype(np.uint32)  # finite, positive
    f = np.concatenate([wide.astype(np.float32), bits.view(np.float32), -bits.view(np.float32)])
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.f64_to_bf16(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, want)


def test_silu_closed_forms():
    l3 = math.log(3.0)
    assert O.silu(l3) == pytest.approx(0.75 * l3, rel=4e-16)
    assert O.silu(-l3) == pytest.approx(-0.25 * l3, rel=4e-16)
    assert O.silu(0.0) == 0.0
    assert O.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert abs(O.silu(-60.0)) < 1e-24


def _small(seed, M=5, N=7, K=96):
    rng = np.random.default_rng(seed)
    xq = rng.integers(-127, 128, (M, K), dtype=np.int64).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K), dtype=np.int64).astype(np.int8)
    xd = (rng.random((M, K // 32)) * 0.05).astype(np.float32)
    wd = (rng.random((N, K // 32)) * 0.01).astype(np.float16).view(np.uint16)
    aux = rng.standard_normal((M, N)).astype(np.float32)
    return xq, xd, wq, wd, aux


def test_zero_weights_give_aux():
    xq, xd, wq, wd, aux = _small(1)
    wq[:] = 0
    y = O.linear_epilogue(xq, xd, wq, wd, aux, "add")
    assert np.array_equal(y, aux)
    yb = O.linear_epilogue(xq, xd, wq, wd, aux, "add", out_bf16=True)
    want = torch.from_numpy(aux.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, want)
    assert not np.any(O.linear_epilogue(xq, xd, wq, wd, aux, "silu_mul"))


def test_no_op_equals_the_pinned_product():
    xq, xd, wq, wd, aux = _small(2)
    y = O.linear_epilogue(xq, xd, wq, wd, aux, "none")
    assert np.array_equal(y, O.linear_codes(xq, xd, wq, wd, nthreads=1))


def test_gated_unit_on_the_unit_code_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "q8_0_closed_form.json")))
    M, N, K = g["M"], g["N"], g["K"]
    xq = np.ones((M, K), np.int8)
    wq = np.ones((N, K), np.int8)
    xd = np.array(g["d_x"], np.float32)
    wd = np.array(g["d_w"], np.float32).astype(np.float16).view(np.uint16)
    gate = np.full((M, N), math.log(3.0), np.float32)
    y = O.linear_epilogue(xq, xd, wq, wd, gate, "silu_mul")
    # the gate is fl32(ln 3): silu there is (3/4) fl32(ln 3) up to ~3e-8 relative
    factor = 0.75 * float(np.float32(math.log(3.0)))
    want = np.array(g["y"], np.float64) * factor
    assert np.allclose(y, want, rtol=2e-7, atol=0)


def test_residual_and_gate_index_alignment():
    xq, xd, wq, wd, aux = _small(3, M=4, N=9, K=64)
    base = O.linear_codes(xq, xd, wq, wd, nthreads=1).astype(np.float64)
    y_add = O.linear_epilogue(xq, xd, wq, wd, aux, "add")
    assert np.allclose(y_add, base + aux.astype(np.float64), rtol=1e-6, atol=1e-6)
    # a gate that is zero except at one (row, column) picks exactly that output
    gate = np.zeros_like(aux)
    gate[2, 5] = math.log(3.0)
    y = O.linear_epilogue(xq, xd, wq, wd, gate, "silu_mul")
    mask = np.zeros_like(y, dtype=bool)
    mask[2, 5] = True
    assert not np.any(y[~mask])
    assert y[2, 5] == pytest.approx(base[2, 5] * 0.75 * float(np.float32(math.log(3.0))), rel=1e-6)
