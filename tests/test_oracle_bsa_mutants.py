"""Planted mistakes in the block-sparse attention oracle must fail its pins.

Each case rewrites one line of a private copy of oracle/bsa_oracle.c (on the CPU, in a
temporary directory), builds it, routes oracle/bsa.py to that build and runs the pins of
tests/test_oracle_bsa.py; at least one must fail.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import bsa
from tests import test_oracle_bsa as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "bsa_oracle.c")

PINS = [
    P.test_equal_value_rows_come_back,
    P.test_zero_keys_average_the_visible_values,
    P.test_first_query_sees_only_itself,
    P.test_two_key_closed_form_fixes_the_scale,
    P.test_sharp_softmax_picks_the_best_key,
    P.test_masked_blocks_and_future_tokens_are_invisible,
    P.test_heads_sharing_a_kv_head_agree,
    P.test_dense_causal_mask_is_library_causal_attention,
    P.test_block_sparse_is_library_attention_under_the_block_mask,
]

MUTANTS = [
    ("causal excludes the query itself", "j < (kb + 1) * OBSA_B && j <= t;", "j < (kb + 1) * OBSA_B && j < t;"),
    ("scale 1/d", "s[n] = dot / sqrt((double)d);", "s[n] = dot / (double)d;"),
    ("kv head h mod Hkv", "int64_t hk = h / (H / Hkv);", "int64_t hk = h % Hkv;"),
    ("block start off by one", "for (int64_t j = kb * OBSA_B; j < (kb + 1) * OBSA_B && j <= t; ++j) {",
     "for (int64_t j = kb * OBSA_B + 1; j < (kb + 1) * OBSA_B && j <= t; ++j) {"),
    ("value of the next key", "const uint16_t *vj = v + (hk * T + idx[i]) * d;",
     "const uint16_t *vj = v + (hk * T + (idx[i] + 1 < T ? idx[i] + 1 : idx[i])) * d;"),
    ("weights not normalised", "double p = s[i] / l;", "double p = s[i];"),
    ("softmax of the negated scores", "s[i] = exp(s[i] - mx);", "s[i] = exp(mx - s[i]);"),
    ("query block from the wrong head", "int32_t e = row_ptr[h * nqb + qb]; e < row_ptr[h * nqb + qb + 1]",
     "int32_t e = row_ptr[qb]; e < row_ptr[qb + 1]"),
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
def test_bsa_mutant_is_caught(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    tmp = tempfile.mkdtemp(prefix="obsamut_")
    try:
        lib = _build_mutant(tmp, old, new)
        caught = False
        with bsa.use_library(lib):
            for pin in PINS:
                try:
                    pin()
                except AssertionError:
                    caught = True
                    break
        assert caught, f"no pin caught the planted mistake: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
