"""Every prefill-sized configuration compared with the CPU oracle on ALL outputs.

The 9B-class and 27B-class prefill projections and every distinct projection shape of the
dense-layer sweep at M = 2048 and M = 8192 run through the library's public call
(q8_linear, bf16 activations) at their full sizes; the oracle (oracle/q8_oracle.c,
multithreaded over output rows) evaluates every output of the same layer from the same
codes, and the two are compared element by element within the library's tolerance
(tests/gpu_util.py).  Weight codes and scales are checked bit for bit first.  One more
test takes the exact int32 block sums of the tensor-core kernel over the 27B up-projection's
whole output tile schedule (M = 8192, N = 17408) and compares them bit for bit.

These tests hold the oracle busy for minutes on the host; they carry the `fullsize`
marker besides `gpu` so that a quick run can deselect them (-m "gpu and not fullsize").
"""
import os

import numpy as np
import pytest

import workloads
from oracle import oracle as O
from tests.gpu_util import assert_close, dev_tensor

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as m
    torch.cuda.set_device(0)
    return m


def _weights(q8, wl, p):
    W = wl.make_weights(p)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(dev_tensor(W, torch))
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(Wd.cpu().numpy().view(np.uint16), Wd_ref)
    return Wq_ref, Wd_ref, Wq, Wd


def _full_case(q8, wl, p, mi, weights):
    Wq_ref, Wd_ref, Wq, Wd = weights
    x, _ = wl.make_act(p, mi)
    M = x.shape[0]
    y = q8.q8_linear(dev_tensor(x, torch), Wq, Wd).cpu().numpy()
    xq_ref, xd_ref = O.quantize_act(x, bf16=True)
    del x
    y_ref = O.linear_codes(xq_ref, xd_ref, Wq_ref, Wd_ref, nthreads=os.cpu_count() or 1)
    assert_close(y, y_ref, f"{wl.name}/{wl.projections[p].name} M={M}, all {y.size} outputs")


@pytest.mark.parametrize("name,p", [("prefill9b", 0), ("prefill9b", 1), ("prefill27b", 0),
                                    ("prefill27b", 1)])
def test_prefill_every_output(q8, name, p):
    wl = workloads.WORKLOADS[name]
    _full_case(q8, wl, p, 0, _weights(q8, wl, p))
    assert q8.q8_device_error() == 0


def test_sweep_large_m_every_output(q8):
    """The distinct projection shapes of the sweep (q/k/v/o 5120x5120, gate/up 5120x17408,
    down 17408x5120, GDN in-proj 5120x10240) at M = 2048 and M = 8192."""
    wl = workloads.WORKLOADS["sweep"]
    seen = set()
    for p, proj in enumerate(wl.projections):
        if (proj.K, proj.N) in seen:
            continue
        seen.add((proj.K, proj.N))
        weights = _weights(q8, wl, p)
        for mi, M in enumerate(wl.Ms):
            if M >= 2048:
                _full_case(q8, wl, p, mi, weights)
    assert q8.q8_device_error() == 0


def test_block_sums_over_the_27b_tile_schedule(q8):
    """Exact int32 block sums of the tensor-core kernel on the 27B up-projection's output
    shape (M = 8192 tokens, N = 17408 weight rows: every tile of that schedule), two Q8_0
    blocks deep, bit for bit against the oracle."""
    rng = np.random.default_rng(31)
    M, N, K = 8192, 17408, 64
    xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
    wq = rng.integers(-127, 128, (N, K), dtype=np.int8)
    xq[:8, :] = 127
    wq[:8, :] = -127                       # extreme blocks: isum = -516128
    ref = O.block_sums(xq, wq)
    got = q8.q8_block_sums(dev_tensor(xq, torch), dev_tensor(wq, torch), path="tensor").cpu().numpy()
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)
