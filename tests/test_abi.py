"""The C ABI without a GPU: the library loads, exports every function include/q8.h
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as q8
    return q8.lib()


def _declared():
    txt = open(os.path.join(ROOT, "include", "q8.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(q8_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"q8_quantize_weights", "q8_quantize_act", "q8_linear"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_exported_symbols_are_declared():
    import subprocess
    import q8_int8_block_gb300 as q8
    out = subprocess.run(["nm", "-D", "--defined-only", q8.lib_path()], capture_output=True,
                         text=True).stdout
    exported = sorted(set(re.findall(r" T (q8_[a-z0-9_]+)$", out, flags=re.M)))
    assert exported == _declared()


def test_status_strings_and_version(L):
    import q8_int8_block_gb300 as q8
    for code in range(10):
        assert L.q8_status_string(code)
    assert q8.q8_version().count(".") == 2


FAKE = 0x10000  # aligned, non-null, never dereferenced: every call below fails validation first
P = ctypes.c_void_p


def test_null_pointers_rejected(L):
    assert L.q8_linear(None, P(FAKE), P(FAKE), P(FAKE), 1, 1, 32, None) == 1
    assert L.q8_linear(P(FAKE), None, P(FAKE), P(FAKE), 1, 1, 32, None) == 1
    assert L.q8_linear_ex(P(FAKE), 1, P(FAKE), None, P(FAKE), 1, 1, 32, 0, None, 0, None) == 1
    assert L.q8_quantize_weights(None, P(FAKE), P(FAKE), 4, 32, None) == 1
    assert L.q8_quantize_act(P(FAKE), 0, None, P(FAKE), 4, 32, None) == 1
    assert L.q8_block_sums(P(FAKE), P(FAKE), None, 1, 1, 32, 0, None) == 1


@pytest.mark.parametrize("M,N,K", [(1, 1, 33), (1, 1, 16), (-1, 4, 32), (4, -2, 32), (4, 4, -32),
                                   (1 << 31, 1, 32), (1, 1, 1 << 40)])
def test_bad_shapes_rejected(L, M, N, K):
    assert L.q8_linear(P(FAKE), P(FAKE), P(FAKE), P(FAKE), M, N, K, None) == 2
    assert L.q8_block_sums(P(FAKE), P(FAKE), P(FAKE), M, N, K, 0, None) == 2


def test_misaligned_pointers_rejected(L):
    for bad in range(4):
        ptrs = [P(FAKE)] * 4
        ptrs[bad] = P(FAKE + 8)
        assert L.q8_linear(ptrs[0], ptrs[1], ptrs[2], ptrs[3], 2, 2, 64, None) == 3
    assert L.q8_quantize_act(P(FAKE + 2), 1, P(FAKE), P(FAKE), 1, 32, None) == 3


def test_bad_dtype_and_path_rejected(L):
    assert L.q8_quantize_act(P(FAKE), 7, P(FAKE), P(FAKE), 1, 32, None) == 4
    assert L.q8_linear_ex(P(FAKE), 2, P(FAKE), P(FAKE), P(FAKE), 1, 1, 32, 0, None, 0, None) == 4
    assert L.q8_linear_ex(P(FAKE), 1, P(FAKE), P(FAKE), P(FAKE), 1, 1, 32, 9, None, 0, None) == 4


def test_valid_call_without_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover real calls")
    # arguments pass validation; the device check then fails without launching anything
    st = L.q8_linear(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 2, 2, 64, None)
    assert st in (6, 7)
    assert L.q8_last_cuda_error()


def test_fused_entry_rejects_bad_arguments(L):
    F = L.q8_linear_fused
    ok = [P(FAKE), 1, None, 1e-6, P(FAKE), P(FAKE), 1, P(FAKE), P(FAKE + 0x1000), 0, 2, 2, 64, 0, None,
          0, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return F(*a)
    assert call(a6=3) == 4            # unknown epilogue
    assert call(a9=2) == 4            # unknown output type
    assert call(a1=5) == 4            # unknown activation type
    assert call(a7=None) == 1         # residual / gate without aux
    assert call(a7=P(FAKE + 4)) == 3  # misaligned aux
    assert call(a8=None) == 1
    assert call(a12=33) == 2
    assert call(a2=P(FAKE + 4)) == 3  # misaligned norm weight
    for eps in (0.0, -1e-6, float("nan"), float("inf")):
        assert call(a2=P(FAKE), a3=eps) == 9
    # aux (M*N floats) overlapping y: in place, bfloat16 y in place, and a partial overlap
    # (64 x 64 floats of aux reach 16 KB past it, y starts 4 KB in)
    assert call(a8=P(FAKE)) == 9
    assert call(a8=P(FAKE), a9=1) == 9
    assert call(a8=P(FAKE + 0x1000), a10=64, a11=64) == 9
    assert call(a7=P(FAKE + 0x1000), a8=P(FAKE), a10=64, a11=64) == 9


def test_rmsnorm_quantizer_rejects_bad_arguments(L):
    Q = L.q8_quantize_act_rmsnorm
    ok = [P(FAKE), 1, P(FAKE), 1e-6, P(FAKE), P(FAKE), P(FAKE), 4, 64, None]
    for i, v, want in ((1, 3, 4), (3, 0.0, 9), (3, float("nan"), 9), (2, None, 1), (6, None, 1),
                       (2, P(FAKE + 8), 3), (8, 48, 2)):
        a = list(ok)
        a[i] = v
        assert Q(*a) == want, (i, v)


def test_kv3_codec_rejects_bad_arguments(L):
    E, D = L.q8_kv3_encode, L.q8_kv3_decode
    E.argtypes = [P, ctypes.c_int, P, P, ctypes.c_int64, P]
    D.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int64, P]
    assert E(P(FAKE), 2, P(FAKE), P(FAKE), 4, None) == 4
    assert E(P(FAKE), 1, P(FAKE), P(FAKE), -1, None) == 2
    assert E(None, 1, P(FAKE), P(FAKE), 4, None) == 1
    assert E(P(FAKE), 1, P(FAKE), P(FAKE + 4), 4, None) == 3
    assert D(P(FAKE), P(FAKE), P(FAKE), 3, 4, None) == 4
    assert D(P(FAKE), None, P(FAKE), 1, 4, None) == 1
    assert D(P(FAKE + 8), P(FAKE), P(FAKE), 1, 4, None) == 3
    assert D(P(FAKE), P(FAKE), P(FAKE), 1, 1 << 50, None) == 2


def test_prepared_entry_rejects_bad_arguments(L):
    W = L.q8_weights_to_f16
    W.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, P]
    assert W(None, P(FAKE), 4, 64, None) == 1
    assert W(P(FAKE), P(FAKE + 2), 4, 64, None) == 3
    assert W(P(FAKE), P(FAKE), 4, 33, None) == 2
    F = L.q8_linear_prepared
    F.argtypes = [P, ctypes.c_int, P, ctypes.c_float, P, P, ctypes.c_int, P, P, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_size_t, P]
    ok = [P(FAKE), 1, None, 1e-6, P(FAKE), P(FAKE), 0, None, P(FAKE), 0, 2, 2, 64, None, 0, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return F(*a)
    assert call(a4=None) == 1          # no prepared weights
    assert call(a6=5) == 4             # unknown epilogue
    assert call(a4=P(FAKE + 8)) == 3   # misaligned prepared weights
    assert call(a12=40) == 2


def test_bsa_entry_rejects_bad_arguments(L):
    F = L.q8_bsa_attention
    F.argtypes = [P, P, P, P, P, ctypes.c_int64, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, P]
    ok = [P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 4, P(FAKE), 0, 4, 2, 128, 128, None]

    def call(i, val):
        a = list(ok)
        a[i] = val
        return F(*a)
    assert call(7, 5) == 4            # output type
    assert call(11, 64) == 2          # head dim other than 128
    assert call(10, 100) == 2         # T not a multiple of 64
    assert call(9, 3) == 2            # H not a multiple of Hkv
    a = list(ok)
    a[8], a[10] = 1 << 22, 1 << 10    # H * T = 2^32: beyond the tiles' 32-bit row coordinates
    assert F(*a) == 2
    assert call(0, None) == 1
    assert call(4, None) == 1         # nnz > 0 without col_idx
    assert call(1, P(FAKE + 2)) == 3
    assert call(3, P(FAKE + 2)) == 3   # row_ptr not on an int32 boundary
    assert call(4, P(FAKE + 1)) == 3   # col_idx likewise
