"""q8_linear_noalloc: the tensor-core Q8_0 linear layer for callers that cannot allocate
device memory during a call (a framework whose device memory all comes from its own fixed
pool, or a serving step that must never call cudaMalloc, which synchronizes the device and
can fail with out-of-memory).  Its scratch is a static device array inside the library.

These tests call it through the C ABI (ctypes) and compare it with the existing entry point
q8_linear_ex on the tensor path, within the same tolerance as the other parity tests, on
calls in a row (so leftover scratch from one call cannot leak into the next), and check
that shapes too large for the array are refused before anything runs.
"""
import ctypes

import numpy as np
import pytest

import workloads
from tests.gpu_util import assert_close, dev_tensor

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as m
    torch.cuda.set_device(0)
    return m


def _noalloc(q8, x, Wq, Wd):
    M, K = x.shape
    N = Wq.shape[0]
    y = torch.full((M, N), float("nan"), device="cuda")
    stream = P(torch.cuda.current_stream().cuda_stream)
    st = q8.lib().q8_linear_noalloc(P(x.data_ptr()), 1 if x.dtype == torch.bfloat16 else 0,
                                    P(Wq.data_ptr()), P(Wd.data_ptr()), P(y.data_ptr()), M, N, K,
                                    stream)
    assert st == 0, q8.lib().q8_status_string(st)
    return y


def test_noalloc_matches_existing_entry_point_on_calls_in_a_row(q8):
    rng = np.random.default_rng(2024)
    cases = [(200, 1000, 1024, True), (64, 300, 512, False), (200, 1000, 1024, True)]
    weights = {}
    for M, N, K, bf16 in cases:
        if (N, K) not in weights:
            W = workloads.weights(rng, N, K)
            weights[(N, K)] = q8.q8_quantize_weights(dev_tensor(W, torch))
        Wq, Wd = weights[(N, K)]
        x, _ = workloads.activations(rng, M, K, bf16=bf16, outlier_frac=0.01)
        xt = dev_tensor(x, torch)
        y = _noalloc(q8, xt, Wq, Wd)
        y_ref = q8.q8_linear_ex(xt, Wq, Wd, path="tensor")
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), y_ref.cpu().numpy(), f"noalloc M={M} N={N} K={K}")


def test_noalloc_refuses_shapes_beyond_its_scratch(q8):
    fake = P(0x10000)  # never dereferenced: the size check comes first
    limit = q8.NOALLOC_SCRATCH_BYTES
    M, N, K = 1024, 16384, 4096  # 2*N*K alone is 128 MiB
    assert 2 * N * K > limit
    st = q8.lib().q8_linear_noalloc(fake, 1, fake, fake, fake, M, N, K, None)
    assert st == 5  # Q8_ERR_NOMEM
