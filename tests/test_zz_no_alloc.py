"""q8_linear_noalloc: the tensor-core Q8_0 linear layer for callers that cannot allocate
device memory during a call (a framework whose device memory all comes from its own fixed
pool, or a serving step that must never call cudaMalloc, which synchronizes the device and
can fail with out-of-memory).  Its scratch is a static device array inside the library.

These tests call it through the C ABI (ctypes) and compare it with the CPU oracle within
the library's tolerance, on calls in a row (so leftover scratch from one call cannot leak
into the next), including calls on both sides of q8_release(); they check that the
library's device error word stays clear, and that shapes too large for the array are
refused before anything runs.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from oracle import oracle as O
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


def _case(q8, rng, M, N, K, bf16):
    """Seeded inputs on the device, plus the oracle's y from the same codes."""
    W = workloads.weights(rng, N, K)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(dev_tensor(W, torch))
    x, _ = workloads.activations(rng, M, K, bf16=bf16, outlier_frac=0.01)
    y_ref = O.linear(x, Wq_ref, Wd_ref, bf16=bf16)
    return dev_tensor(x, torch), Wq, Wd, y_ref


def test_noalloc_matches_oracle_on_calls_in_a_row(q8):
    rng = np.random.default_rng(2024)
    cases = [_case(q8, rng, 200, 1000, 1024, True), _case(q8, rng, 64, 300, 512, False)]
    for i, (xt, Wq, Wd, y_ref) in enumerate(cases + cases[:1]):
        y = _noalloc(q8, xt, Wq, Wd)
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), y_ref, f"noalloc call {i}")
    assert q8.q8_device_error() == 0


def test_noalloc_across_release(q8):
    """q8_release() drops the looked-up device address of the array (and every other
    context-bound cache); the next call looks it up again and still matches the oracle."""
    rng = np.random.default_rng(77)
    xt, Wq, Wd, y_ref = _case(q8, rng, 130, 520, 768, True)
    y0 = _noalloc(q8, xt, Wq, Wd)
    torch.cuda.synchronize()
    assert_close(y0.cpu().numpy(), y_ref, "before q8_release")
    q8.q8_release()
    y1 = _noalloc(q8, xt, Wq, Wd)
    torch.cuda.synchronize()
    assert_close(y1.cpu().numpy(), y_ref, "after q8_release")
    assert q8.q8_device_error() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(q8):
    fake = P(0x10000)  # never dereferenced: the size check comes first
    limit = q8.NOALLOC_SCRATCH_BYTES
    M, N, K = 1024, 16384, 4096  # 2*N*K alone is 128 MiB
    assert 2 * N * K > limit
    st = q8.lib().q8_linear_noalloc(fake, 1, fake, fake, fake, M, N, K, None)
    assert st == 5  # Q8_ERR_NOMEM
