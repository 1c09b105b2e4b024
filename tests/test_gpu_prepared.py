"""The prepared-weights path (q8_weights_to_f16 + q8_linear_prepared): the widened codes are
the exact binary16 values of the int8 codes, and the layer gives the same bits as
q8_linear_fused on the tensor-core path (the same kernels on the same values), with and
without split-K, on a stream-K partial wave, and with the fused neighbours; and matches the
oracle within the layer tolerance."""
import numpy as np
import pytest

import workloads
from oracle import oracle as O
from tests.gpu_util import assert_close, dev_tensor, sample_indices

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


def test_widening_is_exact(q8):
    rng = np.random.default_rng(1)
    Wq = rng.integers(-127, 128, (300, 544), dtype=np.int64).astype(np.int8)
    B16 = q8.q8_weights_to_f16(T(Wq)).cpu().numpy().view(np.uint16)
    assert np.array_equal(B16, Wq.astype(np.float16).view(np.uint16))
    # every byte value in every position of the 16-byte pieces the pass converts
    allc = np.tile(np.arange(-128, 128, dtype=np.int64).astype(np.int8), 33).reshape(33, 256)
    B16 = q8.q8_weights_to_f16(T(allc)).cpu().numpy().view(np.uint16)
    assert np.array_equal(B16, allc.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(130, 300, 96), (128, 256, 4096), (257, 513, 1056),
                                   (129, 19556, 544), (64, 1000, 512)])
def test_same_bits_as_the_tensor_path(q8, M, N, K):
    rng = np.random.default_rng(M + N)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, outlier_frac=0.02)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    B16 = q8.q8_weights_to_f16(Wq)
    xt = T(x)
    a = q8.q8_linear_fused(xt, Wq, Wd, path="tensor")
    b = q8.q8_linear_prepared(xt, B16, Wd)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    g = torch.randn((M, N), device="cuda")
    gamma = torch.rand(K, device="cuda") + 0.5
    a = q8.q8_linear_fused(xt, Wq, Wd, epi="silu_mul", aux=g, out_dtype=torch.bfloat16,
                           path="tensor", norm_weight=gamma)
    b = q8.q8_linear_prepared(xt, B16, Wd, epi="silu_mul", aux=g, out_dtype=torch.bfloat16,
                              norm_weight=gamma)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert q8.q8_device_error() == 0


def test_matches_the_oracle_and_caller_workspace(q8):
    rng = np.random.default_rng(3)
    M, N, K = 300, 700, 2048
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, outlier_frac=0.02)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    ref = O.linear(x, Wq_ref, Wd_ref, bf16=True)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    B16 = q8.q8_weights_to_f16(Wq)
    need = q8.q8_linear_prepared_workspace_size(M, N, K)
    assert need < q8.q8_linear_workspace_size(M, N, K, "tensor")   # no widening scratch
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = q8.q8_linear_prepared(T(x), B16, Wd, workspace=ws)
    assert_close(y.cpu().numpy(), ref, "prepared")
    with pytest.raises(q8.Q8Error) as e:                            # one byte short
        q8.q8_linear_prepared(T(x), B16, Wd, workspace=ws[:need - 1])
    assert e.value.status == 5
    assert q8.q8_device_error() == 0


def test_full_size_prefill(q8):
    wl = workloads.WORKLOADS["prefill9b"]
    W = wl.make_weights(0)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    B16 = q8.q8_weights_to_f16(Wq)
    x, _ = wl.make_act(0, 0)
    y = q8.q8_linear_prepared(T(x), B16, Wd).cpu().numpy()
    xq_ref, xd_ref = O.quantize_act(x, bf16=wl.bf16)
    M, N = y.shape
    rows, cols = sample_indices(np.random.default_rng(5), M, N, 3000)
    ref = O.linear_codes_at(xq_ref, xd_ref, Wq_ref, Wd_ref, rows, cols)
    assert_close(y[rows, cols], ref, "prepared prefill9b up (sampled)")
    assert q8.q8_device_error() == 0
