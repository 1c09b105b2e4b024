"""The build's register pin for kernels that resize registers with setmaxnreg: the compiled
register count must equal the one the kernel's split assumes (else the build stops), and the
library as built passes that check (CPU only: nvcc cross-compiles)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_module():
    spec = importlib.util.spec_from_file_location("_q8_build_t", os.path.join(ROOT, "q8_int8_block_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_register_pin_accepts_only_the_assumed_count():
    b = _build_module()
    src = os.path.join(ROOT, "q8_int8_block_gb300", "csrc", "q8_gemm.cu")
    report = ("ptxas info    : Compiling entry function '_ZN2q8_gemm_tc_kernelILb0ELb0EE' for 'sm_103a'\n"
              "ptxas info    : Used {} registers, used 1 barriers\n")
    b._check_reg_pin(src, report.format(168))
    with pytest.raises(RuntimeError):
        b._check_reg_pin(src, report.format(160))
    with pytest.raises(RuntimeError):
        b._check_reg_pin(src, "no report")


def test_the_gemm_as_built_has_the_assumed_register_count():
    b = _build_module()
    src = os.path.join(ROOT, "q8_int8_block_gb300", "csrc", "q8_gemm.cu")
    obj = b._compile(src, ())   # raises if ptxas allocated another count
    assert os.path.exists(obj)
