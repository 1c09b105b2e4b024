"""Python binding of libq8 (include/q8.h): the Q8_0 block-quantized linear layer on GB300.

Argument marshalling only: every step of the layer runs in the CUDA library.  Tensors
are torch tensors on the current CUDA device (torch provides device memory and streams);
each function passes raw pointers, sizes and the current stream to the C ABI and raises
Q8Error on a non-OK status.  There is no CPU fallback: if libq8.so is missing, importing
this package fails.

    Wq, Wd = q8_quantize_weights(W)              # W float32 [N,K] -> int8 [N,K], fp16 bits [N,K/32]
    xq, xd = q8_quantize_act(x)                  # x bf16/float32 [M,K] -> int8 [M,K], float32 [M,K/32]
    y = q8_linear(x, Wq, Wd)                     # x bf16 [M,K] -> float32 [M,N]
    y = q8_linear_ex(x, Wq, Wd, path="tensor", workspace=ws)
    y = q8_linear_fused(x, Wq, Wd, epi="silu_mul", aux=gate, out_dtype=torch.bfloat16)
    y = q8_linear_fused(h, Wq, Wd, norm_weight=g, norm_eps=1e-6)   # RMSNorm(h) . W^T
    xq, xd, r = q8_quantize_act_rmsnorm(h, g, 1e-6)
    B16 = q8_weights_to_f16(Wq)                        # once per weight matrix
    y = q8_linear_prepared(x, B16, Wd)                 # tensor-core path, no per-call widening
    o = q8_bsa_attention(q, k, v, row_ptr, col_idx)    # block-sparse causal attention
    codes, scales = q8_kv3_encode(kv)                  # kv [..., 128] -> 3-bit codes + scales
    kv_hat = q8_kv3_decode(codes, scales, torch.bfloat16)
    isum = q8_block_sums(xq, Wq, path="decode")  # int32 [M,N,K/32]
"""
import ctypes
import os

import torch

__all__ = ["Q8Error", "q8_quantize_weights", "q8_quantize_act", "q8_quantize_act_rmsnorm",
           "q8_linear", "q8_linear_ex", "q8_kv3_encode", "q8_kv3_decode", "KV3_GROUP",
           "q8_weights_to_f16", "q8_linear_prepared", "q8_linear_prepared_workspace_size",
           "q8_bsa_attention",
           "q8_linear_fused", "EPILOGUES",
           "q8_linear_workspace_size", "q8_block_sums", "q8_device_error", "q8_release",
           "q8_set_timing_events", "q8_linear_noalloc", "NOALLOC_SCRATCH_BYTES",
           "q8_version", "lib_path", "QK", "PATHS"]

QK = 32
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libq8.so")

STATUS = {0: "Q8_OK", 1: "Q8_ERR_NULL", 2: "Q8_ERR_SHAPE", 3: "Q8_ERR_ALIGN", 4: "Q8_ERR_DTYPE",
          5: "Q8_ERR_NOMEM", 6: "Q8_ERR_CUDA", 7: "Q8_ERR_DEVICE", 8: "Q8_ERR_CAPTURE",
          9: "Q8_ERR_VALUE"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
PATHS = {"auto": 0, "decode": 1, "tensor": 2, "batch": 3, "dp4a": 4}
EPILOGUES = {"none": 0, "add": 1, "silu_mul": 2}


class Q8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _L.q8_status_string(status).decode()
        if status == 6:
            msg += ": " + _L.q8_last_cuda_error().decode()
        super().__init__(f"{what}: {STATUS.get(status, status)} ({msg})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libq8.so is not built ({_LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(_LIB_PATH)
    p, i64, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    sigs = {
        "q8_quantize_weights": [p, p, p, i64, i64, p],
        "q8_quantize_act": [p, i32, p, p, i64, i64, p],
        "q8_linear": [p, p, p, p, i64, i64, i64, p],
        "q8_linear_ex": [p, i32, p, p, p, i64, i64, i64, i32, p, sz, p],
        "q8_block_sums": [p, p, p, i64, i64, i64, i32, p],
        "q8_linear_noalloc": [p, i32, p, p, p, i64, i64, i64, p],
        "q8_linear_fused": [p, i32, p, f32, p, p, i32, p, p, i32, i64, i64, i64, i32, p, sz, p],
        "q8_quantize_act_rmsnorm": [p, i32, p, f32, p, p, p, i64, i64, p],
        "q8_kv3_encode": [p, i32, p, p, i64, p],
        "q8_kv3_decode": [p, p, p, i32, i64, p],
        "q8_weights_to_f16": [p, p, i64, i64, p],
        "q8_bsa_attention": [p, p, p, p, p, i64, p, i32, i64, i64, i64, i64, p],
        "q8_linear_prepared": [p, i32, p, f32, p, p, i32, p, p, i32, i64, i64, i64, p, sz, p],
    }
    for name, args in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = i32
    L.q8_set_timing_events.argtypes = [p, p, i32]
    L.q8_set_timing_events.restype = i32
    L.q8_linear_workspace_size.argtypes = [i64, i64, i64, i32]
    L.q8_linear_workspace_size.restype = sz
    L.q8_linear_prepared_workspace_size.argtypes = [i64, i64, i64]
    L.q8_linear_prepared_workspace_size.restype = sz
    L.q8_device_error.argtypes = [ctypes.POINTER(i32)]
    L.q8_device_error.restype = ctypes.c_uint32
    L.q8_status_string.argtypes = [i32]
    L.q8_status_string.restype = ctypes.c_char_p
    L.q8_last_cuda_error.argtypes = []
    L.q8_last_cuda_error.restype = ctypes.c_char_p
    L.q8_release.argtypes = []
    L.q8_release.restype = None
    L.q8_version.argtypes = []
    L.q8_version.restype = ctypes.c_char_p
    return L


_L = _load()


def lib_path() -> str:
    return _LIB_PATH


def lib():
    return _L


def _check(status: int, what: str):
    if status != 0:
        raise Q8Error(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# the current stream's handle without building a torch Stream object (a few microseconds per
# call otherwise); torch has long provided the query, the fallback covers a build without it
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _RAW_STREAM is not None:
            return ctypes.c_void_p(_RAW_STREAM(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _key(table, key, name):
    """table[key], or a ValueError naming the accepted keys."""
    if key not in table:
        raise ValueError(f"{name}: expected one of {sorted(table)}, got {key!r}")
    return table[key]


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")


def _on_device(**tensors):
    """Every tensor given (None skipped) is a contiguous CUDA tensor on the current device:
    the library launches there, so a pointer into host memory or another GPU's memory must
    not reach its kernels.  One device query per call."""
    d = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: must be a contiguous CUDA tensor")
        if d is None:
            d = torch.cuda.current_device()
        if t.get_device() != d:
            raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{d} "
                             "(use torch.cuda.device)")


def q8_quantize_weights(W, Wq=None, Wd=None, stream=None):
    """W float32 [N,K] -> (Wq int8 [N,K], Wd int16-stored binary16 bits [N,K/32])."""
    N, K = W.shape
    _need(W, torch.float32, (N, K), "W")
    if Wq is None:
        Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    if Wd is None:
        Wd = torch.empty((N, K // QK), dtype=torch.int16, device=W.device)
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(Wd, torch.int16, (N, K // QK), "Wd")
    _on_device(W=W, Wq=Wq, Wd=Wd)
    _check(_L.q8_quantize_weights(_ptr(W), _ptr(Wq), _ptr(Wd), N, K, _stream(stream)),
           "q8_quantize_weights")
    return Wq, Wd


def q8_quantize_act(x, xq=None, xd=None, stream=None):
    """x bf16 or float32 [M,K] -> (xq int8 [M,K], xd float32 [M,K/32])."""
    M, K = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    _need(x, x.dtype, (M, K), "x")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xd is None:
        xd = torch.empty((M, K // QK), dtype=torch.float32, device=x.device)
    _need(xq, torch.int8, (M, K), "xq")
    _need(xd, torch.float32, (M, K // QK), "xd")
    _on_device(x=x, xq=xq, xd=xd)
    _check(_L.q8_quantize_act(_ptr(x), DTYPES[x.dtype], _ptr(xq), _ptr(xd), M, K, _stream(stream)),
           "q8_quantize_act")
    return xq, xd


def q8_quantize_act_rmsnorm(x, gamma, eps, xq=None, xd=None, r=None, stream=None):
    """RMSNorm fused into the activation quantizer: x bf16/float32 [M,K], gamma float32 [K]
    -> (xq int8 [M,K]: codes of x * gamma, xd float32 [M,K/32]: their scales times r,
    r float32 [M] = 1 / sqrt(mean(x^2) + eps))."""
    M, K = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    _need(x, x.dtype, (M, K), "x")
    _need(gamma, torch.float32, (K,), "gamma")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xd is None:
        xd = torch.empty((M, K // QK), dtype=torch.float32, device=x.device)
    if r is None:
        r = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(xq, torch.int8, (M, K), "xq")
    _need(xd, torch.float32, (M, K // QK), "xd")
    _need(r, torch.float32, (M,), "r")
    _on_device(x=x, gamma=gamma, xq=xq, xd=xd, r=r)
    _check(_L.q8_quantize_act_rmsnorm(_ptr(x), DTYPES[x.dtype], _ptr(gamma), float(eps), _ptr(xq),
                                      _ptr(xd), _ptr(r), M, K, _stream(stream)),
           "q8_quantize_act_rmsnorm")
    return xq, xd, r


def _lin_check(x, Wq, Wd, y):
    M, K = x.shape
    N = Wq.shape[0]
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(Wd, torch.int16, (N, K // QK), "Wd")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, (M, N), "y")
    return M, N, K, y


def q8_linear(x, Wq, Wd, y=None, stream=None):
    """y float32 [M,N] = Q8_0 linear of bf16 x [M,K] (library-owned scratch)."""
    _need(x, torch.bfloat16, tuple(x.shape), "x")
    M, N, K, y = _lin_check(x, Wq, Wd, y)
    _on_device(x=x, Wq=Wq, Wd=Wd, y=y)
    _check(_L.q8_linear(_ptr(x), _ptr(Wq), _ptr(Wd), _ptr(y), M, N, K, _stream(stream)),
           "q8_linear")
    return y


def q8_linear_workspace_size(M, N, K, path="auto") -> int:
    return int(_L.q8_linear_workspace_size(M, N, K, _key(PATHS, path, "path")))


def q8_linear_ex(x, Wq, Wd, y=None, path="auto", workspace=None, stream=None):
    """q8_linear with activation type (bf16/float32), kernel family and caller scratch.
    workspace: a uint8 CUDA tensor of at least q8_linear_workspace_size() bytes, or None
    (then one is allocated here with torch)."""
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    path_id = _key(PATHS, path, "path")
    _need(x, x.dtype, tuple(x.shape), "x")
    M, N, K, y = _lin_check(x, Wq, Wd, y)
    need = q8_linear_workspace_size(M, N, K, path)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _on_device(x=x, Wq=Wq, Wd=Wd, y=y, workspace=workspace)
    _check(_L.q8_linear_ex(_ptr(x), DTYPES[x.dtype], _ptr(Wq), _ptr(Wd), _ptr(y), M, N, K,
                           path_id, _ptr(workspace), nbytes, _stream(stream)), "q8_linear_ex")
    return y


def q8_linear_fused(x, Wq, Wd, epi="none", aux=None, y=None, out_dtype=torch.float32,
                    path="auto", workspace=None, stream=None, norm_weight=None, norm_eps=1e-6):
    """The linear layer with its neighbours fused into it.  norm_weight (float32 [K]): the
    input is RMSNorm(x) with that weight and norm_eps, applied inside the layer's quantizer.
    epi "none": y = x.W^T; "add": y = x.W^T + aux (residual); "silu_mul":
    y = silu(aux) * x.W^T (aux the gate projection's output).  aux float32 [M,N];
    y float32 or bfloat16 [M,N].  workspace None uses the library-owned scratch."""
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    if out_dtype not in DTYPES:
        raise TypeError(f"out_dtype: expected bfloat16 or float32, got {out_dtype}")
    epi_id, path_id = _key(EPILOGUES, epi, "epi"), _key(PATHS, path, "path")
    if epi_id != 0 and aux is None:
        raise ValueError(f"epi {epi!r} needs aux")
    _need(x, x.dtype, tuple(x.shape), "x")
    M, K = x.shape
    N = Wq.shape[0]
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(Wd, torch.int16, (N, K // QK), "Wd")
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _need(y, out_dtype, (M, N), "y")
    if epi_id != 0:
        _need(aux, torch.float32, (M, N), "aux")
    if norm_weight is not None:
        _need(norm_weight, torch.float32, (K,), "norm_weight")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _on_device(x=x, norm_weight=norm_weight, Wq=Wq, Wd=Wd, aux=aux, y=y, workspace=workspace)
    _check(_L.q8_linear_fused(_ptr(x), DTYPES[x.dtype], _ptr(norm_weight), float(norm_eps),
                              _ptr(Wq), _ptr(Wd), epi_id,
                              _ptr(aux), _ptr(y), DTYPES[out_dtype], M, N, K, path_id,
                              _ptr(workspace), nbytes, _stream(stream)), "q8_linear_fused")
    return y


def q8_weights_to_f16(Wq, B16=None, stream=None):
    """Wq int8 [N,K] -> B16 int16-stored binary16 codes [N,K], for q8_linear_prepared."""
    N, K = Wq.shape
    _need(Wq, torch.int8, (N, K), "Wq")
    if B16 is None:
        B16 = torch.empty((N, K), dtype=torch.int16, device=Wq.device)
    _need(B16, torch.int16, (N, K), "B16")
    _on_device(Wq=Wq, B16=B16)
    _check(_L.q8_weights_to_f16(_ptr(Wq), _ptr(B16), N, K, _stream(stream)), "q8_weights_to_f16")
    return B16


def q8_linear_prepared_workspace_size(M, N, K) -> int:
    return int(_L.q8_linear_prepared_workspace_size(M, N, K))


def q8_linear_prepared(x, B16, Wd, epi="none", aux=None, y=None, out_dtype=torch.float32,
                       workspace=None, stream=None, norm_weight=None, norm_eps=1e-6):
    """q8_linear_fused on the tensor-core path with weights widened once by
    q8_weights_to_f16 (no per-call widening)."""
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    if out_dtype not in DTYPES:
        raise TypeError(f"out_dtype: expected bfloat16 or float32, got {out_dtype}")
    epi_id = _key(EPILOGUES, epi, "epi")
    if epi_id != 0 and aux is None:
        raise ValueError(f"epi {epi!r} needs aux")
    _need(x, x.dtype, tuple(x.shape), "x")
    M, K = x.shape
    N = B16.shape[0]
    _need(B16, torch.int16, (N, K), "B16")
    _need(Wd, torch.int16, (N, K // QK), "Wd")
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _need(y, out_dtype, (M, N), "y")
    if epi_id != 0:
        _need(aux, torch.float32, (M, N), "aux")
    if norm_weight is not None:
        _need(norm_weight, torch.float32, (K,), "norm_weight")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _on_device(x=x, norm_weight=norm_weight, B16=B16, Wd=Wd, aux=aux, y=y, workspace=workspace)
    _check(_L.q8_linear_prepared(_ptr(x), DTYPES[x.dtype], _ptr(norm_weight), float(norm_eps),
                                 _ptr(B16), _ptr(Wd), epi_id, _ptr(aux), _ptr(y),
                                 DTYPES[out_dtype], M, N, K, _ptr(workspace), nbytes,
                                 _stream(stream)), "q8_linear_prepared")
    return y


def q8_bsa_attention(q, k, v, row_ptr, col_idx, out_dtype=torch.float32, o=None, stream=None):
    """Block-sparse causal attention: q [H,T,128], k and v [Hkv,T,128] bfloat16; row_ptr
    int32 [H*T/64+1], col_idx int32 [nnz] (the listed 64-token key blocks of each head's
    64-token query block) -> o [H,T,128] of out_dtype."""
    H, T, d = q.shape
    Hkv = k.shape[0]
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, (H if name == "q" else Hkv, T, d), name)
    _need(row_ptr, torch.int32, (H * (T // 64) + 1,), "row_ptr")
    if col_idx.dim() != 1:
        raise ValueError("col_idx: a 1-D int32 CUDA tensor")
    _need(col_idx, torch.int32, (col_idx.numel(),), "col_idx")
    if out_dtype not in DTYPES:
        raise TypeError(f"out_dtype: expected bfloat16 or float32, got {out_dtype}")
    if o is None:
        o = torch.empty((H, T, d), dtype=out_dtype, device=q.device)
    _need(o, out_dtype, (H, T, d), "o")
    _on_device(q=q, k=k, v=v, row_ptr=row_ptr, col_idx=col_idx, o=o)
    _check(_L.q8_bsa_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(row_ptr), _ptr(col_idx),
                               col_idx.numel(), _ptr(o), DTYPES[out_dtype], H, Hkv, T, d,
                               _stream(stream)), "q8_bsa_attention")
    return o


KV3_GROUP = 128


def q8_kv3_encode(x, codes=None, scales=None, stream=None):
    """3-bit KV-cache codec, encoder: x bf16/float32 [..., 128*k] (contiguous) ->
    (codes int32 [groups, 12] holding the uint32 code words, scales float32 [groups]), one
    group per 128 consecutive elements.  Reinterpret codes with .view(torch.int32) as needed."""
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    if x.numel() % KV3_GROUP:
        raise ValueError("x: a contiguous CUDA tensor of whole 128-element groups")
    _need(x, x.dtype, tuple(x.shape), "x")
    n = x.numel() // KV3_GROUP
    if codes is None:
        codes = torch.empty((n, 12), dtype=torch.int32, device=x.device)
    if scales is None:
        scales = torch.empty((n,), dtype=torch.float32, device=x.device)
    _need(codes, torch.int32, (n, 12), "codes")
    _need(scales, torch.float32, (n,), "scales")
    _on_device(x=x, codes=codes, scales=scales)
    _check(_L.q8_kv3_encode(_ptr(x), DTYPES[x.dtype], _ptr(codes), _ptr(scales), n, _stream(stream)),
           "q8_kv3_encode")
    return codes, scales


def q8_kv3_decode(codes, scales, out_dtype=torch.bfloat16, out=None, stream=None):
    """3-bit KV-cache codec, decoder: (codes int32 [groups, 12], scales float32 [groups]) ->
    out [groups, 128] of out_dtype (bfloat16 or float32)."""
    n = codes.shape[0]
    _need(codes, torch.int32, (n, 12), "codes")
    _need(scales, torch.float32, (n,), "scales")
    if out_dtype not in DTYPES:
        raise TypeError(f"out_dtype: expected bfloat16 or float32, got {out_dtype}")
    if out is None:
        out = torch.empty((n, KV3_GROUP), dtype=out_dtype, device=codes.device)
    _need(out, out_dtype, (n, KV3_GROUP), "out")
    _on_device(codes=codes, scales=scales, out=out)
    _check(_L.q8_kv3_decode(_ptr(codes), _ptr(scales), _ptr(out), DTYPES[out_dtype], n,
                            _stream(stream)), "q8_kv3_decode")
    return out


NOALLOC_SCRATCH_BYTES = 64 << 20


def q8_linear_noalloc(x, Wq, Wd, y=None, stream=None):
    """Tensor-core Q8_0 linear that allocates no device memory: its scratch is a static
    device array of NOALLOC_SCRATCH_BYTES in the library (see include/q8.h).  For callers
    whose memory is owned by a fixed pool or whose step must not allocate.  Calls that
    overlap on the GPU share that array and race; make the first call on a device before
    any stream capture."""
    if x.dtype not in DTYPES:
        raise TypeError(f"x: expected bfloat16 or float32, got {x.dtype}")
    _need(x, x.dtype, tuple(x.shape), "x")
    M, N, K, y = _lin_check(x, Wq, Wd, y)
    _on_device(x=x, Wq=Wq, Wd=Wd, y=y)
    _check(_L.q8_linear_noalloc(_ptr(x), DTYPES[x.dtype], _ptr(Wq), _ptr(Wd), _ptr(y), M, N, K,
                                _stream(stream)), "q8_linear_noalloc")
    return y


def q8_block_sums(xq, Wq, isum=None, path="auto", stream=None):
    """Exact int32 block sums isum [M,N,K/32] of int8 codes, by the kernel of `path`."""
    path_id = _key(PATHS, path, "path")
    M, K = xq.shape
    N = Wq.shape[0]
    _need(xq, torch.int8, (M, K), "xq")
    _need(Wq, torch.int8, (N, K), "Wq")
    if isum is None:
        isum = torch.empty((M, N, K // QK), dtype=torch.int32, device=xq.device)
    _need(isum, torch.int32, (M, N, K // QK), "isum")
    _on_device(xq=xq, Wq=Wq, isum=isum)
    _check(_L.q8_block_sums(_ptr(xq), _ptr(Wq), _ptr(isum), M, N, K, path_id, _stream(stream)),
           "q8_block_sums")
    return isum


def q8_device_error() -> int:
    """Synchronizes the device and returns (and clears) the device error word (0 = none)."""
    st = ctypes.c_int(0)
    word = _L.q8_device_error(ctypes.byref(st))
    _check(st.value, "q8_device_error")
    return int(word)


def q8_set_timing_events(starts=None, stops=None):
    """Timing hook: events (torch.cuda.Event(enable_timing=True)) recorded around the main
    kernel of each later q8_linear / q8_linear_ex call, cycling through the list; under
    graph capture they become event nodes.  No arguments: switch off."""
    if not starts:
        _check(_L.q8_set_timing_events(None, None, 0), "q8_set_timing_events")
        return
    assert len(starts) == len(stops)
    for e in list(starts) + list(stops):  # make sure the CUDA events exist
        if e.cuda_event == 0:
            e.record()
    arr = ctypes.c_void_p * len(starts)
    a = arr(*[e.cuda_event for e in starts])
    b = arr(*[e.cuda_event for e in stops])
    _check(_L.q8_set_timing_events(a, b, len(starts)), "q8_set_timing_events")


def q8_release():
    _L.q8_release()


def q8_version() -> str:
    return _L.q8_version().decode()
