"""numpy front end of the 3-bit KV-cache codec oracle (oracle/kv3_oracle.c).

TEST INFRASTRUCTURE ONLY (tests, the package smoke check and the benchmark's CPU-baseline
leg).  The codec's readings K1-K6 are stated in kv3_oracle.c.
"""
import contextlib
import ctypes

import numpy as np

from . import build as _build

D = 128      # elements per group
WORDS = 12   # 3-bit codes of a group, as uint32 words
LEVELS = (0.2451, 0.7560, 1.3440, 2.1520)       # Max (1960), 8-level unit-Gaussian quantizer
THRESHOLDS = (0.5006, 1.0500, 1.7480)

_lib = None


def _load(path):
    L = ctypes.CDLL(path)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    L.okv3_fwht.argtypes = [p]
    L.okv3_fwht.restype = None
    L.okv3_encode_group.argtypes = [p, p, p]
    L.okv3_encode_group.restype = None
    L.okv3_decode_group.argtypes = [p, ctypes.c_float, p]
    L.okv3_decode_group.restype = None
    L.okv3_encode.argtypes = [p, ctypes.c_int, i64, p, p]
    L.okv3_encode.restype = None
    L.okv3_decode.argtypes = [p, p, i64, p]
    L.okv3_decode.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build_kv3())
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Route the front end to another build (planted-mistake tests)."""
    global _lib
    old = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = old


def _ptr(a):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def fwht(v):
    """Unnormalised fast Walsh-Hadamard transform of one 128-vector in binary32 (K2)."""
    a = np.ascontiguousarray(v, dtype=np.float32).copy()
    assert a.shape == (D,)
    lib().okv3_fwht(_ptr(a))
    return a


def encode(x, bf16=False):
    """x [n,128] float32 (or bfloat16 bits as uint16) -> (words uint32 [n,12], scales float32 [n])."""
    x = np.ascontiguousarray(x, dtype=np.uint16 if bf16 else np.float32)
    n = x.shape[0]
    assert x.shape == (n, D)
    words = np.zeros((n, WORDS), np.uint32)
    scales = np.zeros(n, np.float32)
    lib().okv3_encode(_ptr(x), 1 if bf16 else 0, n, _ptr(words), _ptr(scales))
    return words, scales


def decode(words, scales):
    """(words [n,12], scales [n]) -> float32 [n,128]."""
    words = np.ascontiguousarray(words, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    n = words.shape[0]
    out = np.empty((n, D), np.float32)
    lib().okv3_decode(_ptr(words), _ptr(scales), n, _ptr(out))
    return out


def codes(words):
    """Unpack [n,12] words into [n,128] 3-bit codes (bits [3i, 3i + 3) of the stream, K5)."""
    w = np.ascontiguousarray(words, dtype=np.uint32)
    bits = np.unpackbits(w.view(np.uint8), axis=1, bitorder="little")[:, :3 * D]
    b = bits.reshape(w.shape[0], D, 3).astype(np.uint8)
    return b[:, :, 0] | (b[:, :, 1] << 1) | (b[:, :, 2] << 2)
