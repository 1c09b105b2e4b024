"""Parity of the RMSNorm prologue (RMSNorm fused into the activation quantizer) with the
oracle, standalone (q8_quantize_act_rmsnorm) and inside every kernel family
(q8_linear_fused with norm_weight).

Codes are bit-exact: they depend on fl32(x * gamma) only.  r and the scales it carries
are binary32 on the GPU and binary64 in the oracle: relative 1e-5 (a fixed-order binary32
sum of K squares is within about (K/256 + 16) 2^-24 of the exact one).  Outputs y: the
layer tolerance (binary32), or the bfloat16 rule of the epilogue tests.
"""
import numpy as np
import pytest

import workloads
from oracle import oracle as O
from tests.gpu_util import assert_close, dev_tensor
from tests.test_gpu_epilogue import assert_bf16_close, torch_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-6


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


def _hidden(rng, M, K, bf16=True):
    """Hidden states: N(0,1) with outlier channels, one all-zero row and one row scaled by
    1e3 (the norm must remove the row's magnitude)."""
    x, _ = workloads.activations(rng, M, K, bf16=False, outlier_frac=0.02)
    if M > 2:
        x[1] = 0.0
        x[2] *= np.float32(1e3)
    return workloads.bf16_bits_from_f32(x) if bf16 else x


def _gamma(rng, K):
    return (0.25 + 1.5 * rng.random(K)).astype(np.float32)


@pytest.mark.parametrize("M,K,bf16", [(1, 4096, True), (7, 96, False), (64, 5120, True),
                                      (300, 17408, True), (33, 512, False)])
def test_rmsnorm_quantizer(q8, M, K, bf16):
    rng = np.random.default_rng(M + K)
    x = _hidden(rng, M, K, bf16)
    g = _gamma(rng, K)
    xq_ref, xd_ref, r_ref = O.rmsnorm_quantize_act(x, g, EPS, bf16=bf16)
    xq, xd, r = q8.q8_quantize_act_rmsnorm(T(x), T(g), EPS)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    r = r.cpu().numpy().astype(np.float64)
    assert np.allclose(r, r_ref, rtol=1e-5, atol=0)
    want = xd_ref.astype(np.float64) * r_ref[:, None]
    assert np.allclose(xd.cpu().numpy().astype(np.float64), want, rtol=1e-5, atol=0)


CASES = [
    ("decode", 1, 300, 4096), ("decode", 5, 257, 4128), ("decode", 8, 129, 96),
    ("batch", 16, 1000, 512), ("batch", 33, 77, 1024),
    ("tensor", 130, 300, 96), ("tensor", 128, 256, 4096), ("tensor", 257, 513, 1056),
    ("dp4a", 65, 129, 96), ("dp4a", 200, 300, 4128),
    ("auto", 1, 256, 512), ("auto", 40, 256, 1024), ("auto", 300, 700, 512),
]


@pytest.mark.parametrize("op", ["none", "silu_mul"])
@pytest.mark.parametrize("path,M,N,K", CASES)
def test_normalised_layer_matches_oracle(q8, path, M, N, K, op):
    rng = np.random.default_rng(M * 7 + N + K)
    W = workloads.weights(rng, N, K)
    x = _hidden(rng, M, K)
    g = _gamma(rng, K)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    xq_ref, xd_ref, r_ref = O.rmsnorm_quantize_act(x, g, EPS, bf16=True)
    aux = (rng.standard_normal((M, N)) * 2.5).astype(np.float32)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    xt, gt, at = T(x), T(g), T(aux)
    aux_arg = None if op == "none" else at
    what = f"{path} norm+{op} M={M} N={N} K={K}"

    y = q8.q8_linear_fused(xt, Wq, Wd, epi=op, aux=aux_arg, path=path, norm_weight=gt, norm_eps=EPS)
    ref = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, aux, op, rowscale=r_ref)
    assert_close(y.cpu().numpy(), ref, what)
    for r in range(min(M, 4)):  # the zero row and the 1e3 row on their own scale
        if np.max(np.abs(ref[r])) > 0:
            assert_close(y[r].cpu().numpy(), ref[r], f"{what} row {r}")
    y2 = q8.q8_linear_fused(xt, Wq, Wd, epi=op, aux=aux_arg, path=path, norm_weight=gt, norm_eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), what + " (not deterministic)"

    yb = q8.q8_linear_fused(xt, Wq, Wd, epi=op, aux=aux_arg, path=path, norm_weight=gt,
                            norm_eps=EPS, out_dtype=torch.bfloat16)
    refb = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, aux, op, out_bf16=True, rowscale=r_ref)
    assert_bf16_close(torch_bits(yb), refb, what + " bf16")
    assert q8.q8_device_error() == 0


def test_unit_norm_weight_matches_scaled_plain_layer(q8):
    """With gamma = 1 the codes are the plain quantizer's, so the normalised layer is the
    plain layer times r per row (up to binary32 rounding)."""
    rng = np.random.default_rng(31)
    M, N, K = 6, 500, 2048
    W = workloads.weights(rng, N, K)
    x = _hidden(rng, M, K)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    ones = torch.ones(K, device="cuda")
    for path in ("decode", "batch", "tensor", "dp4a"):
        y = q8.q8_linear_fused(T(x), Wq, Wd, path=path, norm_weight=ones, norm_eps=EPS).cpu().numpy()
        y0 = q8.q8_linear_ex(T(x), Wq, Wd, path=path).cpu().numpy().astype(np.float64)
        _, _, r = q8.q8_quantize_act_rmsnorm(T(x), ones, EPS)
        assert_close(y, y0 * r.cpu().numpy().astype(np.float64)[:, None], path)


@pytest.mark.parametrize("name,p", [("decode", 0), ("prefill9b", 0)])
def test_normalised_layer_full_size(q8, name, p):
    wl = workloads.WORKLOADS[name]
    W = wl.make_weights(p)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    rng = np.random.default_rng(41)
    for mi in range(len(wl.Ms)):
        x, _ = wl.make_act(p, mi)
        M, K = x.shape
        g = _gamma(rng, K)
        y = q8.q8_linear_fused(T(x), Wq, Wd, norm_weight=T(g), norm_eps=EPS).cpu().numpy()
        rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 4)]))
        xq_ref, xd_ref, r_ref = O.rmsnorm_quantize_act(x[rows], g, EPS, bf16=wl.bf16)
        ref = O.linear_epilogue(xq_ref, xd_ref, Wq_ref, Wd_ref, rowscale=r_ref)
        assert_close(y[rows], ref, f"{name} M={M} normalised (rows {rows.tolist()})")
    assert q8.q8_device_error() == 0
