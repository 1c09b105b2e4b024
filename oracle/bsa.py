"""numpy front end of the block-sparse attention oracle (oracle/bsa_oracle.c).

TEST INFRASTRUCTURE ONLY (tests, the package smoke check and the benchmark's CPU-baseline
leg).  The readings A1-A4 are stated in bsa_oracle.c.
"""
import contextlib
import ctypes

import numpy as np

from . import build as _build

B = 64   # tokens per block

_lib = None


def _load(path):
    L = ctypes.CDLL(path)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    L.obsa_attention.argtypes = [p, p, p, i64, i64, i64, i64, p, p, p]
    L.obsa_attention.restype = None
    L.obsa_attention_at.argtypes = [p, p, p, i64, i64, i64, i64, p, p, p, p, i64, p]
    L.obsa_attention_at.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build_bsa())
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


def _args(q, k, v, row_ptr, col_idx):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    H, T, d = q.shape
    Hkv = k.shape[0]
    assert k.shape == (Hkv, T, d) and v.shape == (Hkv, T, d) and H % Hkv == 0 and T % B == 0
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    assert rp.shape == (H * (T // B) + 1,)
    return q, k, v, H, Hkv, T, d, rp, ci


def attention(q, k, v, row_ptr, col_idx):
    """q [H,T,d], k, v [Hkv,T,d] bf16 bits (uint16); CSR block mask -> o float32 [H,T,d]."""
    q, k, v, H, Hkv, T, d, rp, ci = _args(q, k, v, row_ptr, col_idx)
    o = np.empty((H, T, d), np.float32)
    lib().obsa_attention(_ptr(q), _ptr(k), _ptr(v), H, Hkv, T, d, _ptr(rp), _ptr(ci), _ptr(o))
    return o


def attention_at(q, k, v, row_ptr, col_idx, heads, tokens):
    """Only the queries (heads[s], tokens[s]) -> float32 [n, d]."""
    q, k, v, H, Hkv, T, d, rp, ci = _args(q, k, v, row_ptr, col_idx)
    hs = np.ascontiguousarray(heads, dtype=np.int64)
    ts = np.ascontiguousarray(tokens, dtype=np.int64)
    o = np.empty((hs.shape[0], d), np.float32)
    lib().obsa_attention_at(_ptr(q), _ptr(k), _ptr(v), H, Hkv, T, d, _ptr(rp), _ptr(ci),
                            _ptr(hs), _ptr(ts), hs.shape[0], _ptr(o))
    return o
