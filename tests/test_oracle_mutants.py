"""Planted mistakes in the oracle must fail its pins.

Each case rewrites one line of a private copy of oracle/q8_oracle.c (on the CPU, in a
temporary directory), builds it, routes the oracle's Python front end to that build and
runs the pin tests; at least one pin must fail.  This checks the pins themselves.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import oracle as O
from tests import test_oracle_epilogue as E
from tests import test_oracle_norm as R
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "q8_oracle.c")

PINS = [
    P.test_f32_to_f16_matches_numpy_rne,
    P.test_golden_tie_blocks,
    P.test_roundtrip_bound_and_extreme_codes,
    P.test_roundtrip_bound_with_binary16_weight_scale,
    P.test_all_zero_block_gives_zero_scale_and_codes,
    P.test_block_sums_brute_force,
    P.test_closed_form_unit_codes,
    lambda: P.test_linear_within_quantization_bound(5, 7, 96, False),
    lambda: P.test_linear_within_quantization_bound(16, 40, 512, True),
    P.test_bf16_path_equals_widened_f32_path,
    E.test_bf16_rounding_hand_worked,
    E.test_silu_closed_forms,
    E.test_zero_weights_give_aux,
    E.test_residual_and_gate_index_alignment,
    E.test_gated_unit_on_the_unit_code_closed_form,
    R.test_constant_rows_closed_form,
    lambda: R.test_two_level_rows(1.0, 3.0, 1e-6),
    R.test_gamma_on_one_block_scales_only_that_block,
    R.test_gamma_zero_on_odd_columns,
    lambda: R.test_normalised_layer_within_the_quantization_bound(5, 7, 96, False),
]

# (name, text in the source, replacement)
MUTANTS = [
    ("half-to-even codes", "float r = roundf(v[j] / d);", "float r = rintf(v[j] / d);"),
    ("truncated codes", "float r = roundf(v[j] / d);", "float r = truncf(v[j] / d);"),
    ("reciprocal multiply", "float r = roundf(v[j] / d);", "float r = roundf(v[j] * (1.0f / d));"),
    ("scale amax/128", "float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    ("signed amax", "float a = fabsf(v[j]);", "float a = v[j];"),
    ("binary16 truncation", "double mant = nearbyint((2.0 * fr - 1.0) * 1024.0);",
     "double mant = floor((2.0 * fr - 1.0) * 1024.0);"),
    ("dropped last block", "for (int64_t b = 0; b < nb; ++b) {\n        int64_t s = 0;",
     "for (int64_t b = 0; b + 1 < nb; ++b) {\n        int64_t s = 0;"),
    ("wrong block index in sums", "isum[(m * N + n) * nb + b] = (int32_t)s;",
     "isum[(n * M + m) * nb + b] = (int32_t)s;"),
    ("scale from the wrong block", "acc += oq8_f16_to_f64(wd_row[b]) * (double)xd_row[b] * (double)s;",
     "acc += oq8_f16_to_f64(wd_row[0]) * (double)xd_row[b] * (double)s;"),
    ("sign flip", "acc += oq8_f16_to_f64(wd_row[b]) * (double)xd_row[b] * (double)s;",
     "acc -= oq8_f16_to_f64(wd_row[b]) * (double)xd_row[b] * (double)s;"),
    ("bf16 widening off by a byte", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 8;"),
    ("zero block gets scale 1", "*d32 = 0.0f;", "*d32 = 1.0f;"),
    ("bf16 output truncated", "double q = nearbyint(ldexp(2.0 * m, 7));",
     "double q = floor(ldexp(2.0 * m, 7));"),
    ("residual subtracted", "return acc + (double)aux[i];", "return acc - (double)aux[i];"),
    ("silu of the negated gate", "double oq8_silu(double g) { return g / (1.0 + exp(-g)); }",
     "double oq8_silu(double g) { return g / (1.0 + exp(g)); }"),
    ("gate from the wrong element", "return oq8_silu((double)aux[i]) * acc;",
     "return oq8_silu((double)aux[i / 2]) * acc;"),
    ("norm mean over K - 1", "double mean = K > 0 ? ss / (double)K : 0.0;",
     "double mean = K > 1 ? ss / (double)(K - 1) : 0.0;"),
    ("norm eps outside the root", "r[m] = 1.0 / sqrt(mean + eps);", "r[m] = 1.0 / (sqrt(mean) + eps);"),
    ("norm factor not inverted", "r[m] = 1.0 / sqrt(mean + eps);", "r[m] = sqrt(mean + eps);"),
    ("norm mean of (x * gamma)^2", "double a = (double)oq8_act_value(x, dtype, m * K + k);",
     "double a = (double)oq8_act_value(x, dtype, m * K + k) * gamma[k];"),
    ("norm gamma one column off", "u[j] = oq8_act_value(x, dtype, m * K + k) * gamma[k];",
     "u[j] = oq8_act_value(x, dtype, m * K + k) * gamma[(k + 1) % K];"),
    ("norm row factor dropped", "acc = acc * rowscale[m];", "acc = acc;"),
]


def _build_mutant(tmp, old, new):
    src = open(SRC).read()
    assert old in src, old
    path = os.path.join(tmp, "mut.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = os.path.join(tmp, "libmut.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                    path, "-o", lib, "-lm"], check=True)
    return lib


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    tmp = tempfile.mkdtemp(prefix="oq8mut_")
    try:
        lib = _build_mutant(tmp, old, new)
        failures = []
        with O.use_library(lib):
            for pin in PINS:
                try:
                    pin()
                except AssertionError as e:  # the pin caught it
                    failures.append(getattr(pin, "__name__", "pin"))
                    break
        assert failures, f"no pin caught the planted mistake: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
