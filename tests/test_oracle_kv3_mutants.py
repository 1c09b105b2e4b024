"""Planted mistakes in the KV-codec oracle must fail its pins.

Each case rewrites one line of a private copy of oracle/kv3_oracle.c (on the CPU, in a
temporary directory), builds it, routes oracle/kv3.py to that build and runs the pins of
tests/test_oracle_kv3.py; at least one must fail.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import kv3
from tests import test_oracle_kv3 as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "kv3_oracle.c")

PINS = [
    P.test_fwht_is_the_sylvester_hadamard_matrix,
    P.test_fwht_twice_is_128_times_identity,
    *[lambda c=c: P.test_decoder_levels_are_the_table(c) for c in range(8)],
    *[lambda k=k: P.test_decision_thresholds_from_the_closed_form(k) for k in range(3)],
    lambda: P.test_unit_vector_codes_layout_and_exact_round_trip(37, -0.5),
    lambda: P.test_unit_vector_codes_layout_and_exact_round_trip(127, 8.0),
    P.test_zero_group,
    P.test_exact_zeros_get_the_positive_code,
    P.test_negative_zero_rotation_output_gets_the_positive_code,
    P.test_scale_is_the_rms_of_the_rotated_group,
    P.test_gaussian_distortion_is_the_lloyd_max_one,
]

MUTANTS = [
    ("butterfly outputs swapped", "a[j] = x + y;\n                a[j + h] = x - y;",
     "a[j] = x - y;\n                a[j + h] = x + y;"),
    ("last stage dropped", "for (int h = 1; h < OKV3_D; h <<= 1)", "for (int h = 1; h < OKV3_D / 2; h <<= 1)"),
    ("mean over 127", "float s = sqrtf(ss / 128.0f);", "float s = sqrtf(ss / 127.0f);"),
    ("sum of |u| instead of squares", "sq[i] = u[i] * u[i];", "sq[i] = fabsf(u[i]);"),
    ("level typo", "{0.2451f, 0.7560f, 1.3440f, 2.1520f}", "{0.2451f, 0.7650f, 1.3440f, 2.1520f}"),
    ("threshold typo", "{0.5006f, 1.0500f, 1.7480f}", "{0.5006f, 1.0050f, 1.7480f}"),
    ("sign on u <= 0", "uint32_t code = (u[i] < 0.0f ? 4u : 0u) | m;", "uint32_t code = (u[i] <= 0.0f ? 4u : 0u) | m;"),
    ("sign from the sign bit", "uint32_t code = (u[i] < 0.0f ? 4u : 0u) | m;",
     "uint32_t code = (signbit(u[i]) ? 4u : 0u) | m;"),
    ("threshold not scaled", "T[k] = okv3_threshold[k] * s;", "T[k] = okv3_threshold[k];"),
    ("bit offset", "int bit = 3 * i;\n        words[bit / 32] |= code << (bit % 32);",
     "int bit = 3 * i + 1;\n        words[bit / 32] |= code << (bit % 32);"),
    ("decode without the 1/128", "out[i] = w[i] / 128.0f;", "out[i] = w[i] / 64.0f;"),
    ("decode without the scale", "w[i] = scale * ((code & 4u) ? -level : level);",
     "w[i] = (code & 4u) ? -level : level;"),
    ("decode sign lost", "w[i] = scale * ((code & 4u) ? -level : level);", "w[i] = scale * level;"),
]


def _build_mutant(tmp, old, new):
    src = open(SRC).read()
    assert old in src, old
    path = os.path.join(tmp, "mut.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = os.path.join(tmp, "libmut.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", path, "-o",
                    lib, "-lm"], check=True)
    return lib


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_kv3_mutant_is_caught(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    tmp = tempfile.mkdtemp(prefix="okv3mut_")
    try:
        lib = _build_mutant(tmp, old, new)
        caught = False
        with kv3.use_library(lib):
            for pin in PINS:
                try:
                    pin()
                except AssertionError:
                    caught = True
                    break
        assert caught, f"no pin caught the planted mistake: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
