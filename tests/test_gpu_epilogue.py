"""Parity of the fused epilogue (q8_linear_fused: residual add, SiLU-gated unit, bfloat16
output) with the oracle, on every kernel family.

binary32 outputs: the tolerance of tests/gpu_util.py (the kernels evaluate the epilogue
in binary32, the oracle in binary64 with one rounding; expf and the division add a few
binary32 ulps, far inside it).
bfloat16 outputs: (a) bit-exact against round-to-nearest-even of the same path's binary32
output (the rounding itself); (b) against the oracle's once-rounded bfloat16, at most one
bfloat16 ulp plus the binary32 tolerance apart (a binary32 sum within the tolerance of
the exact one can sit on the other side of a rounding boundary), and equal almost
everywhere.
"""
import numpy as np
import pytest

import workloads
from oracle import oracle as O
from tests.gpu_util import REL_MAX, assert_close, dev_tensor

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as m
    torch.cuda.set_device(0)
    return m


def T(a):
    return dev_tensor(a, torch)


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def torch_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bf16_close(got_bits, ref_bits, what=""):
    a = bf16_bits_to_f64(got_bits)
    b = bf16_bits_to_f64(ref_bits)
    scale = np.max(np.abs(b)) if b.size else 0.0
    bound = 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 2 * REL_MAX * scale
    bad = np.abs(a - b) > bound
    assert not np.any(bad), f"{what}: {np.count_nonzero(bad)} outputs beyond one bf16 ulp"
    same = np.count_nonzero(a == b) / max(a.size, 1)
    assert same >= 0.99, f"{what}: only {same:.4f} of bf16 outputs equal"


def _inputs(rng, M, N, K, op):
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=True, outlier_frac=0.02)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    xq_ref, xd_ref = O.quantize_act(x, bf16=True)
    base = O.linear_codes(xq_ref, xd_ref, Wq_ref, Wd_ref)
    s = float(np.std(base)) or 1.0
    if op == "silu_mul":      # a gate projection's output: a few units wide, both signs
        aux = (rng.standard_normal((M, N)) * 2.5).astype(np.float32)
    else:                     # a residual stream on the scale of the product
        aux = (rng.standard_normal((M, N)) * s).astype(np.float32)
    return W, x, xq_ref, xd_ref, Wq_ref, Wd_ref, aux


CASES = [
    ("decode", 1, 300, 4096), ("decode", 5, 257, 4128), ("decode", 8, 129, 96),
    ("batch", 16, 1000, 512), ("batch", 33, 77, 1024), ("batch", 64, 2433, 256),
    ("tensor", 130, 300, 96),     # one K split
    ("tensor", 128, 256, 4096),   # split-K: partials reduced by a second kernel
    ("tensor", 257, 513, 1056),   # ragged tiles, split-K
    ("dp4a", 65, 129, 96), ("dp4a", 200, 300, 4128),
    ("auto", 1, 256, 512), ("auto", 40, 256, 1024), ("auto", 300, 700, 512),
]


@pytest.mark.parametrize("op", ["none", "add", "silu_mul"])
@pytest.mark.parametrize("path,M,N,K", CASES)
def test_fused_epilogue_matches_oracle(q8, path, M, N, K, op):
    rng = np.random.default_rng(M * 13 + N * 3 + K + len(op))
    W, x, xq_ref, xd_ref, Wq_ref, Wd_ref, aux = _inputs(rng, M, N, K, op)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    xt, at = T(x), T(aux)
    aux_arg = None if op == "none" else at
    what = f"{path} {op} M={M} N={N} K={K}"

    y32 = q8.q8_linear_fused(xt, Wq, Wd, epi=op, aux=aux_arg, path=path)
    ref32 = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, aux, op)
    assert_close(y32.cpu().numpy(), ref32, what + " f32")

    y16 = q8.q8_linear_fused(xt, Wq, Wd, epi=op, aux=aux_arg, out_dtype=torch.bfloat16, path=path)
    got = torch_bits(y16)
    assert np.array_equal(got, torch_bits(y32.to(torch.bfloat16))), what + " bf16 rounding"
    ref16 = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, aux, op, out_bf16=True)
    assert_bf16_close(got, ref16, what + " bf16")
    assert q8.q8_device_error() == 0


def test_fused_none_equals_the_plain_layer(q8):
    rng = np.random.default_rng(21)
    for path, M, N, K in (("decode", 3, 500, 1024), ("batch", 20, 700, 2048),
                          ("tensor", 128, 256, 4096), ("dp4a", 70, 300, 512)):
        W = workloads.weights(rng, N, K)
        x, _ = workloads.activations(rng, M, K)
        Wq, Wd = q8.q8_quantize_weights(T(W))
        a = q8.q8_linear_ex(T(x), Wq, Wd, path=path)
        b = q8.q8_linear_fused(T(x), Wq, Wd, path=path)
        torch.cuda.synchronize()
        assert torch.equal(a, b), path


def test_fused_caller_workspace_matches_library_scratch(q8):
    rng = np.random.default_rng(22)
    M, N, K = 24, 700, 2048
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    g = torch.randn((M, N), device="cuda")
    for path in ("batch", "tensor", "dp4a"):
        ws = torch.empty(q8.q8_linear_workspace_size(M, N, K, path), dtype=torch.uint8, device="cuda")
        a = q8.q8_linear_fused(T(x), Wq, Wd, epi="silu_mul", aux=g, path=path, workspace=ws)
        b = q8.q8_linear_fused(T(x), Wq, Wd, epi="silu_mul", aux=g, path=path)
        torch.cuda.synchronize()
        assert torch.equal(a, b), path


def test_fused_empty_sum_applies_the_epilogue_to_zero(q8):
    M, N = 3, 37
    rng = np.random.default_rng(23)
    aux = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    x = torch.ones((M, 0), dtype=torch.bfloat16, device="cuda")
    Wq = torch.zeros((N, 0), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((N, 0), dtype=torch.int16, device="cuda")
    xq = np.zeros((M, 0), np.int8)
    xd = np.zeros((M, 0), np.float32)
    wq = np.zeros((N, 0), np.int8)
    wd = np.zeros((N, 0), np.uint16)
    for op in ("none", "add", "silu_mul"):
        for bf16 in (False, True):
            y = q8.q8_linear_fused(x, Wq, Wd, epi=op, aux=None if op == "none" else T(aux),
                                   out_dtype=torch.bfloat16 if bf16 else torch.float32)
            ref = O.linear_epilogue(xq, xd, wq, wd, aux, op, out_bf16=bf16)
            if bf16:
                assert np.array_equal(bf16_bits_to_f64(torch_bits(y)), bf16_bits_to_f64(ref)), op
            else:
                assert np.array_equal(y.cpu().numpy(), ref), op
    assert q8.q8_device_error() == 0


def test_fused_bf16_output_stays_inside_its_buffer(q8):
    rng = np.random.default_rng(24)
    for (M, N, K, path) in ((5, 77, 256, "decode"), (131, 259, 96, "tensor"), (13, 77, 256, "batch"),
                            (128, 250, 4096, "tensor"), (65, 129, 96, "dp4a")):
        W = workloads.weights(rng, N, K)
        x, _ = workloads.activations(rng, M, K)
        Wq, Wd = q8.q8_quantize_weights(T(W))
        pad = 64  # bf16 guard on each side (16-byte aligned slice)
        big = torch.full((M * N + 2 * pad,), float("nan"), device="cuda", dtype=torch.bfloat16)
        y = big[pad:pad + M * N].view(M, N)
        r = torch.randn((M, N), device="cuda")
        q8.q8_linear_fused(T(x), Wq, Wd, epi="add", aux=r, y=y, out_dtype=torch.bfloat16, path=path)
        torch.cuda.synchronize()
        assert torch.isnan(big[:pad]).all() and torch.isnan(big[pad + M * N:]).all(), path
        assert torch.isfinite(y).all(), path


@pytest.mark.parametrize("name,p", [("prefill9b", 0), ("decode", 0)])
def test_fused_gated_unit_full_size(q8, name, p):
    """The gated unit at full size: sampled rows of the whole [M,N] output against the
    oracle on those rows."""
    wl = workloads.WORKLOADS[name]
    W = wl.make_weights(p)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    mi = len(wl.Ms) - 1 if name == "decode" else 0
    x, _ = wl.make_act(p, mi)
    M, N = x.shape[0], Wq_ref.shape[0]
    rng = np.random.default_rng(25)
    gate = (rng.standard_normal((M, N)) * 2.5).astype(np.float32)
    y = q8.q8_linear_fused(T(x), Wq, Wd, epi="silu_mul", aux=T(gate), out_dtype=torch.bfloat16)
    got = torch_bits(y)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 4)]))
    xq_ref, xd_ref = O.quantize_act(x[rows], bf16=wl.bf16)
    ref = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, gate[rows], "silu_mul", out_bf16=True)
    assert_bf16_close(got[rows], ref, f"{name} gated unit (rows {rows.tolist()})")
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("op,bf16,M,N,K", [("silu_mul", True, 129, 19556, 544),
                                           ("add", False, 129, 19556, 544),
                                           ("silu_mul", True, 300, 26000, 544)])
def test_fused_epilogue_on_stream_k(q8, op, bf16, M, N, K):
    """Partial last waves (154 and 306 tiles on the GPU's 152 SMs): tiles that one CTA covers
    whole apply the epilogue in the GEMM drain, tiles that two stream-K runs share in the
    reduction of their partials; both must match the oracle."""
    rng = np.random.default_rng(77)
    W, x, xq_ref, xd_ref, Wq_ref, Wd_ref, aux = _inputs(rng, M, N, K, op)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    out = torch.bfloat16 if bf16 else torch.float32
    y = q8.q8_linear_fused(T(x), Wq, Wd, epi=op, aux=T(aux), out_dtype=out, path="tensor")
    ref = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, aux, op, out_bf16=bf16)
    if bf16:
        assert_bf16_close(torch_bits(y), ref, f"stream-K {op} bf16")
    else:
        assert_close(y.cpu().numpy(), ref, f"stream-K {op}")
    assert q8.q8_device_error() == 0
