"""numpy front end of the C oracle (oracle/q8_oracle.c).

TEST INFRASTRUCTURE ONLY.  Callers: tests/, the package smoke check and the
benchmark's CPU-baseline leg.  Nothing here touches the CUDA library.

Layouts (all row-major, K contiguous):
    W  float32 [N, K]          Wq int8 [N, K]     Wd uint16 [N, K/32] (binary16 bits)
    x  float32 or bf16-bits    xq int8 [M, K]     xd float32 [M, K/32]
    y  float32 [M, N] = x . W^T through the Q8_0 codes
"""
import ctypes
import os

import numpy as np

from . import build as _build

QK = 32
_lib = None


def _load(path):
    L = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    L.oq8_f32_to_f16.argtypes = [ctypes.c_float]
    L.oq8_f32_to_f16.restype = ctypes.c_uint16
    L.oq8_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oq8_f16_to_f64.restype = ctypes.c_double
    L.oq8_quantize_block.argtypes = [p, p, p]
    L.oq8_quantize_weights.argtypes = [p, i64, i64, p, p]
    L.oq8_quantize_act_f32.argtypes = [p, i64, i64, p, p]
    L.oq8_quantize_act_bf16.argtypes = [p, i64, i64, p, p]
    L.oq8_block_sums.argtypes = [p, p, i64, i64, i64, p]
    L.oq8_linear_codes.argtypes = [p, p, p, p, i64, i64, i64, p, ctypes.c_int]
    L.oq8_linear_codes_at.argtypes = [p, p, p, p, i64, p, p, i64, p]
    L.oq8_linear.argtypes = [p, ctypes.c_int, p, p, p, i64, i64, i64, p, p, ctypes.c_int]
    L.oq8_f64_to_bf16.argtypes = [ctypes.c_double]
    L.oq8_f64_to_bf16.restype = ctypes.c_uint16
    L.oq8_silu.argtypes = [ctypes.c_double]
    L.oq8_silu.restype = ctypes.c_double
    L.oq8_linear_epilogue.argtypes = [p, p, p, p, i64, i64, i64, p, p, ctypes.c_int, ctypes.c_int, p]
    L.oq8_rmsnorm_quantize_act.argtypes = [p, ctypes.c_int, p, ctypes.c_double, i64, i64, p, p, p]
    L.oq8_rmsnorm_quantize_act.restype = None
    L.oq8_linear_epilogue.restype = None
    for f in ("oq8_quantize_block", "oq8_quantize_weights", "oq8_quantize_act_f32",
              "oq8_quantize_act_bf16", "oq8_block_sums", "oq8_linear_codes",
              "oq8_linear_codes_at", "oq8_linear"):
        getattr(L, f).restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


class use_library:
    """Context manager: route this module's calls to another build of the oracle source
    (the mutation tests use it to check that the pins catch planted mistakes)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = _load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def f32_to_f16_bits(v: float) -> int:
    return int(lib().oq8_f32_to_f16(ctypes.c_float(v)))


def f16_bits_to_f64(h: int) -> float:
    return float(lib().oq8_f16_to_f64(ctypes.c_uint16(h)))


def quantize_block(v: np.ndarray):
    """One 32-element block -> (codes int8[32], binary32 scale)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (QK,)
    q = np.zeros(QK, np.int8)
    d = np.zeros(1, np.float32)
    lib().oq8_quantize_block(_ptr(v), _ptr(q), _ptr(d))
    return q, d[0]


def quantize_weights(W: np.ndarray):
    """W float32 [N,K] -> (Wq int8 [N,K], Wd uint16 [N,K/32] binary16 bits)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % QK == 0
    Wq = np.empty((N, K), np.int8)
    Wd = np.empty((N, K // QK), np.uint16)
    lib().oq8_quantize_weights(_ptr(W), N, K, _ptr(Wq), _ptr(Wd))
    return Wq, Wd


def quantize_act(x: np.ndarray, bf16: bool = False):
    """x [M,K] (float32, or uint16 bfloat16 bits when bf16=True) -> (xq int8, xd float32)."""
    if bf16:
        x = np.ascontiguousarray(x, dtype=np.uint16)
    else:
        x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % QK == 0
    xq = np.empty((M, K), np.int8)
    xd = np.empty((M, K // QK), np.float32)
    f = lib().oq8_quantize_act_bf16 if bf16 else lib().oq8_quantize_act_f32
    f(_ptr(x), M, K, _ptr(xq), _ptr(xd))
    return xq, xd


def block_sums(xq: np.ndarray, Wq: np.ndarray):
    """-> isum int32 [M, N, K/32], exact."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    M, K = xq.shape
    N = Wq.shape[0]
    out = np.empty((M, N, K // QK), np.int32)
    lib().oq8_block_sums(_ptr(xq), _ptr(Wq), M, N, K, _ptr(out))
    return out


def linear_codes(xq, xd, Wq, Wd, nthreads: int = 0):
    """y float32 [M,N] from codes and scales (binary64 sum, one final rounding)."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint16)
    M, K = xq.shape
    N = Wq.shape[0]
    y = np.empty((M, N), np.float32)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    lib().oq8_linear_codes(_ptr(xq), _ptr(xd), _ptr(Wq), _ptr(Wd), M, N, K, _ptr(y), nthreads)
    return y


def linear_codes_at(xq, xd, Wq, Wd, rows, cols):
    """Sampled outputs y[rows[i], cols[i]]."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    assert rows.shape == cols.shape
    out = np.empty(rows.shape, np.float32)
    lib().oq8_linear_codes_at(_ptr(xq), _ptr(xd), _ptr(Wq), _ptr(Wd), xq.shape[1], _ptr(rows),
                              _ptr(cols), rows.size, _ptr(out))
    return out


def linear(x, Wq, Wd, bf16: bool = False, nthreads: int = 0):
    """The whole layer from raw activations: quantize x, then the rescaled block sums."""
    if bf16:
        x = np.ascontiguousarray(x, dtype=np.uint16)
    else:
        x = np.ascontiguousarray(x, dtype=np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint16)
    M, K = x.shape
    N = Wq.shape[0]
    xq = np.empty((M, K), np.int8)
    xd = np.empty((M, K // QK), np.float32)
    y = np.empty((M, N), np.float32)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    lib().oq8_linear(_ptr(x), 1 if bf16 else 0, _ptr(Wq), _ptr(Wd), _ptr(y), M, N, K, _ptr(xq),
                     _ptr(xd), nthreads)
    return y


EPILOGUES = {"none": 0, "add": 1, "silu_mul": 2}


def f64_to_bf16(v: float) -> int:
    """binary64 -> bfloat16 bits, round to nearest even."""
    return int(lib().oq8_f64_to_bf16(float(v)))


def silu(g: float) -> float:
    return float(lib().oq8_silu(float(g)))


def linear_epilogue(xq, xd, Wq, Wd, aux=None, op="none", out_bf16=False, rowscale=None):
    """y = op(rowscale[m] * rescaled block sums, aux) in binary64, rounded once to binary32
    or to bfloat16 (returned as uint16 bits).  op: "none", "add" (residual: y = acc + aux)
    or "silu_mul" (gated unit: y = silu(aux) * acc).  rowscale: binary64 [M] (the RMSNorm
    factor r of rmsnorm_quantize_act) or None."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint16)
    M, K = xq.shape
    N = Wq.shape[0]
    a = np.zeros((M, N), np.float32) if aux is None else np.ascontiguousarray(aux, dtype=np.float32)
    y = np.empty((M, N), np.uint16 if out_bf16 else np.float32)
    rs = None if rowscale is None else np.ascontiguousarray(rowscale, dtype=np.float64)
    lib().oq8_linear_epilogue(_ptr(xq), _ptr(xd), _ptr(Wq), _ptr(Wd), M, N, K,
                              None if rs is None else _ptr(rs), _ptr(a),
                              EPILOGUES[op], 1 if out_bf16 else 0, _ptr(y))
    return y


def rmsnorm_quantize_act(x, gamma, eps, bf16=False):
    """RMSNorm fused into the activation quantizer (readings N1-N3 of q8_oracle.c):
    x [M,K] (float32, or bfloat16 bits as uint16 when bf16), gamma [K] float32, eps > 0 ->
    (xq int8 [M,K]: codes of u = fl32(x * gamma), xd_u float32 [M,K/32]: scales of u,
    r float64 [M] = 1 / sqrt(mean(x^2) + eps)).  The activation scale is xd_u * r."""
    x = np.ascontiguousarray(x, dtype=np.uint16 if bf16 else np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    M, K = x.shape
    assert gamma.shape == (K,) and K % QK == 0
    xq = np.empty((M, K), np.int8)
    xd = np.empty((M, K // QK), np.float32)
    r = np.empty(M, np.float64)
    lib().oq8_rmsnorm_quantize_act(_ptr(x), 1 if bf16 else 0, _ptr(gamma), float(eps), M, K,
                                   _ptr(xq), _ptr(xd), _ptr(r))
    return xq, xd, r
