"""Parity of the CUDA library (through its C ABI) with the CPU oracle.

Bit-exact: int8 codes, binary16 weight scales, binary32 activation scales, int32 block sums
(on both kernel families).  Within tolerance (tests/gpu_util.py): binary32 outputs y.
Sizes: small shapes that span several tiles and ragged tails, compared element by element;
and every configured workload at full size, compared on sampled outputs (and on full
outputs where the oracle finishes in seconds).
"""
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


def _crafted_matrix(rows, K, seed):
    """Weights/activations with zero blocks, exact ties, huge and tiny blocks."""
    rng = np.random.default_rng(seed)
    A = workloads.weights(rng, rows, K, std=1.0)
    nb = K // 32
    A[0, :] = 0.0                                   # all-zero row
    if nb > 1:
        A[1, 32:64] = 0.0                           # one zero block
    A[2 % rows, :32] = np.float32(0.5) * np.arange(-16, 16, dtype=np.float32)  # ties
    A[3 % rows, :32] = np.float32(127.0) * np.sign(np.arange(32) - 15.5).astype(np.float32)
    A[4 % rows, :32] = A[4 % rows, :32] * np.float32(1e-30)   # tiny normal-range block
    A[5 % rows, :32] = A[5 % rows, :32] * np.float32(1e30)    # huge block
    A[6 % rows, :32] = np.float32(3e-43) * np.linspace(-1, 1, 32, dtype=np.float32)  # subnormal
    return A


# ------------------------------------------------------------------------------------ #
# quantizers: bit-exact                                                                 #
# ------------------------------------------------------------------------------------ #

@pytest.mark.parametrize("N,K,crafted", [(256, 512, False), (12288, 4096, False), (61, 96, True),
                                         (7, 17408, True)])
def test_weight_quantizer_bit_exact(q8, N, K, crafted):
    W = _crafted_matrix(N, K, 5) if crafted else workloads.weights(np.random.default_rng(N), N, K)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(Wd.cpu().numpy().view(np.uint16), Wd_ref)


@pytest.mark.parametrize("M,K,bf16,outliers,crafted", [
    (16, 512, False, 0.0, False), (64, 4096, True, 0.0, False), (300, 17408, True, 0.01, False),
    (33, 5120, True, 0.01, False), (9, 96, False, 0.0, True), (9, 96, True, 0.0, True)])
def test_activation_quantizer_bit_exact(q8, M, K, bf16, outliers, crafted):
    if crafted:
        x32 = _crafted_matrix(M, K, 6)
        x = workloads.bf16_bits_from_f32(x32) if bf16 else x32
    else:
        x, _ = workloads.activations(np.random.default_rng(M + K), M, K, bf16=bf16,
                                     outlier_frac=outliers)
    xq_ref, xd_ref = O.quantize_act(x, bf16=bf16)
    xq, xd = q8.q8_quantize_act(T(x))
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(xd.cpu().numpy().view(np.uint32), xd_ref.view(np.uint32))


# ------------------------------------------------------------------------------------ #
# block sums: bit-exact, both kernel families                                          #
# ------------------------------------------------------------------------------------ #

def _codes(rng, rows, K):
    q = rng.integers(-127, 128, size=(rows, K), dtype=np.int8)
    if rows > 2 and K >= 64:
        q[1, :32] = 127           # extreme blocks: sums of +-516128
        q[2, :32] = -127
        q[0, 32:64] = 0
    return q


@pytest.mark.parametrize("path,M,N,K", [
    ("decode", 1, 7, 64), ("decode", 3, 100, 288), ("decode", 8, 33, 4096),
    ("decode", 5, 257, 4128), ("decode", 1, 700, 17408), ("decode", 6, 1500, 4096),
    ("tensor", 16, 256, 512), ("tensor", 130, 300, 96), ("tensor", 1, 1, 32),
    ("tensor", 257, 513, 160), ("tensor", 3, 40, 4096),
    ("batch", 2, 7, 256), ("batch", 5, 300, 512), ("batch", 16, 1000, 4096), ("batch", 33, 257, 768),
    ("batch", 64, 2500, 4096), ("batch", 8, 17408, 256), ("batch", 1, 100, 1024),
    ("batch", 61, 3001, 5120),
    ("dp4a", 1, 1, 32), ("dp4a", 65, 129, 96), ("dp4a", 200, 300, 4128), ("dp4a", 64, 128, 64)])
def test_block_sums_bit_exact(q8, path, M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    xq = _codes(rng, M, K)
    wq = _codes(rng, N, K)
    ref = O.block_sums(xq, wq)
    got = q8.q8_block_sums(T(xq), T(wq), path=path).cpu().numpy()
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------------------------ #
# linear layer: small shapes, element by element                                       #
# ------------------------------------------------------------------------------------ #

@pytest.mark.parametrize("path,M,N,K,bf16", [
    ("decode", 1, 300, 4096, True), ("decode", 2, 257, 4128, True), ("decode", 4, 1000, 512, False),
    ("decode", 2, 64, 17408, True), ("decode", 3, 5, 32, True), ("decode", 7, 129, 96, False),
    ("decode", 1, 5120, 17408, True), ("decode", 4, 3000, 12288, True), ("decode", 8, 2000, 4096, True),
    ("tensor", 16, 256, 512, False), ("tensor", 130, 300, 96, True), ("tensor", 257, 513, 1056, True),
    ("tensor", 128, 256, 4096, True), ("tensor", 1, 17, 32, True), ("tensor", 200, 100, 4128, False),
    ("batch", 2, 300, 4096, True), ("batch", 7, 129, 256, False), ("batch", 16, 1000, 512, True),
    ("batch", 33, 77, 1024, True), ("batch", 64, 2000, 4096, True), ("batch", 17, 40, 17408, True),
    ("batch", 64, 2432, 256, False), ("batch", 9, 2433, 512, True), ("batch", 1, 5, 256, True),
    ("dp4a", 1, 17, 32, True), ("dp4a", 65, 129, 96, False), ("dp4a", 200, 300, 4128, True),
    ("dp4a", 128, 256, 4096, True), ("dp4a", 7, 1000, 17408, True),
    ("auto", 16, 256, 512, False), ("auto", 1, 256, 512, True), ("auto", 40, 256, 1024, True)])
def test_linear_small_shapes(q8, path, M, N, K, bf16):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=bf16, outlier_frac=0.02)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    y_ref = O.linear(x, Wq_ref, Wd_ref, bf16=bf16)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    y = q8.q8_linear_ex(T(x), Wq, Wd, path=path).cpu().numpy()
    assert_close(y, y_ref, f"{path} M={M} N={N} K={K}")
    assert q8.q8_device_error() == 0


def test_crafted_blocks_through_the_layer(q8):
    W = _crafted_matrix(40, 256, 7)
    W[5, :32] = 1.0  # keep the output in a sane range: the huge block stays in x only
    x32 = _crafted_matrix(12, 256, 8)
    x = workloads.bf16_bits_from_f32(x32)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    y_ref = O.linear(x, Wq_ref, Wd_ref, bf16=True)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    for path in ("decode", "tensor"):
        rows = 8 if path == "decode" else 12
        y = q8.q8_linear_ex(T(x[:rows]), Wq, Wd, path=path).cpu().numpy()
        ref = O.linear(x[:rows], Wq_ref, Wd_ref, bf16=True)
        # rows with huge activations dominate max|y|; compare row by row as well
        assert_close(y, ref, path)
        for r in range(rows):
            if np.max(np.abs(ref[r])) > 0:
                assert_close(y[r], ref[r], f"{path} row {r}")


# ------------------------------------------------------------------------------------ #
# full-size workloads                                                                   #
# ------------------------------------------------------------------------------------ #

def _run_case(q8, wl, p, mi, Wq_ref, Wd_ref, Wq, Wd, full_limit=4e9, samples=3000):
    x, _ = wl.make_act(p, mi)
    M, K = x.shape
    N = Wq_ref.shape[0]
    y = q8.q8_linear(T(x), Wq, Wd).cpu().numpy() if wl.bf16 else \
        q8.q8_linear_ex(T(x), Wq, Wd).cpu().numpy()
    xq_ref, xd_ref = O.quantize_act(x, bf16=wl.bf16)
    if M * N * K <= full_limit:
        y_ref = O.linear_codes(xq_ref, xd_ref, Wq_ref, Wd_ref)
        assert_close(y, y_ref, f"{wl.name}/{wl.projections[p].name} M={M}")
    else:
        rows, cols = sample_indices(np.random.default_rng(M + N + K), M, N, samples)
        ref = O.linear_codes_at(xq_ref, xd_ref, Wq_ref, Wd_ref, rows, cols)
        assert_close(y[rows, cols], ref, f"{wl.name}/{wl.projections[p].name} M={M} (sampled)")
        # every row and every column must have been written (NaN-free, not left at zero)
        assert np.all(np.isfinite(y))
        assert np.count_nonzero(np.abs(y).max(axis=1) == 0) == 0
    return y


def _weights(q8, wl, p):
    W = wl.make_weights(p)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(Wd.cpu().numpy().view(np.uint16), Wd_ref)
    return Wq_ref, Wd_ref, Wq, Wd


def test_workload_tiny(q8):
    wl = workloads.WORKLOADS["tiny"]
    _run_case(q8, wl, 0, 0, *_weights(q8, wl, 0))


def test_workload_decode_all_batch_sizes(q8):
    wl = workloads.WORKLOADS["decode"]
    args = _weights(q8, wl, 0)
    for mi in range(len(wl.Ms)):
        _run_case(q8, wl, 0, mi, *args)


@pytest.mark.parametrize("name", ["prefill9b", "prefill27b"])
def test_workload_prefill(q8, name):
    wl = workloads.WORKLOADS[name]
    for p in range(len(wl.projections)):
        _run_case(q8, wl, p, 0, *_weights(q8, wl, p), full_limit=0)


def test_workload_dense_layer_sweep(q8):
    wl = workloads.WORKLOADS["sweep"]
    for p in range(len(wl.projections)):
        args = _weights(q8, wl, p)
        for mi in range(len(wl.Ms)):
            _run_case(q8, wl, p, mi, *args, full_limit=2e8, samples=500)
    assert q8.q8_device_error() == 0


# ------------------------------------------------------------------------------------ #
# API behaviour on the device                                                           #
# ------------------------------------------------------------------------------------ #

def test_library_workspace_matches_caller_workspace_and_is_deterministic(q8):
    rng = np.random.default_rng(12)
    W = workloads.weights(rng, 700, 2048)
    x, _ = workloads.activations(rng, 300, 2048)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    xt = T(x)
    y1 = q8.q8_linear(xt, Wq, Wd)
    y2 = q8.q8_linear_ex(xt, Wq, Wd, path="tensor")
    y3 = q8.q8_linear(xt, Wq, Wd)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(y1, y3)
    for M in (1, 3, 8, 20, 64):
        a = q8.q8_linear(xt[:M].contiguous(), Wq, Wd)
        b = q8.q8_linear(xt[:M].contiguous(), Wq, Wd)
        assert torch.equal(a, b)
    # the batched path with a caller workspace gives the same bits as with the library's
    xb = xt[:24].contiguous()
    ws = torch.empty(q8.q8_linear_workspace_size(24, 700, 2048, "batch"), dtype=torch.uint8,
                     device="cuda")
    a = q8.q8_linear_ex(xb, Wq, Wd, path="batch", workspace=ws)
    b = q8.q8_linear_ex(xb, Wq, Wd, path="batch")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_outputs_stay_inside_their_buffers(q8):
    rng = np.random.default_rng(13)
    for (M, N, K, path) in ((5, 77, 256, "decode"), (131, 259, 96, "tensor"), (13, 77, 256, "batch"),
                            (64, 3001, 512, "batch"), (129, 19556, 544, "tensor")):
        W = workloads.weights(rng, N, K)
        x, _ = workloads.activations(rng, M, K)
        Wq, Wd = q8.q8_quantize_weights(T(W))
        pad = 64  # floats of guard on each side (16-byte aligned slice)
        big = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
        y = big[pad:pad + M * N].view(M, N)
        q8.q8_linear_ex(T(x), Wq, Wd, y=y, path=path)
        torch.cuda.synchronize()
        assert torch.isnan(big[:pad]).all() and torch.isnan(big[pad + M * N:]).all()
        assert torch.isfinite(y).all()


def test_empty_and_zero_sizes(q8):
    Wq = torch.zeros((4, 64), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((4, 2), dtype=torch.int16, device="cuda")
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    assert q8.q8_linear(x, Wq, Wd).shape == (0, 4)
    x = torch.ones((3, 0), dtype=torch.bfloat16, device="cuda")
    y = torch.full((3, 4), 5.0, device="cuda")
    q8.q8_linear(x, torch.zeros((4, 0), dtype=torch.int8, device="cuda"),
                 torch.zeros((4, 0), dtype=torch.int16, device="cuda"), y=y)
    assert torch.count_nonzero(y) == 0   # empty sum
    xq, xd = q8.q8_quantize_act(torch.zeros((0, 32), dtype=torch.float32, device="cuda"))
    assert xq.shape == (0, 32)
    assert q8.q8_device_error() == 0


def test_decode_path_rejects_large_m(q8):
    Wq = torch.zeros((4, 64), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((4, 2), dtype=torch.int16, device="cuda")
    x = torch.zeros((9, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_linear_ex(x, Wq, Wd, path="decode")
    assert e.value.status == 2


def test_batch_path_rejects_unsupported_shapes(q8):
    Wq = torch.zeros((4, 512), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((4, 16), dtype=torch.int16, device="cuda")
    with pytest.raises(q8.Q8Error) as e:   # more than 64 tokens
        q8.q8_linear_ex(torch.zeros((65, 512), dtype=torch.bfloat16, device="cuda"), Wq, Wd,
                        path="batch")
    assert e.value.status == 2
    Wq = torch.zeros((4, 288), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((4, 9), dtype=torch.int16, device="cuda")
    with pytest.raises(q8.Q8Error) as e:   # K not a multiple of 256
        q8.q8_linear_ex(torch.zeros((4, 288), dtype=torch.bfloat16, device="cuda"), Wq, Wd,
                        path="batch")
    assert e.value.status == 2
    assert q8.q8_device_error() == 0


def test_dp4a_path_full_size_prefill(q8):
    """The post's own design (dp4a GEMM) on the 9B-class up-projection, sampled outputs."""
    wl = workloads.WORKLOADS["prefill9b"]
    Wq_ref, Wd_ref, Wq, Wd = _weights(q8, wl, 0)
    x, _ = wl.make_act(0, 0)
    y = q8.q8_linear_ex(T(x), Wq, Wd, path="dp4a").cpu().numpy()
    xq_ref, xd_ref = O.quantize_act(x, bf16=wl.bf16)
    M, N = y.shape
    rows, cols = sample_indices(np.random.default_rng(77), M, N, 3000)
    ref = O.linear_codes_at(xq_ref, xd_ref, Wq_ref, Wd_ref, rows, cols)
    assert_close(y[rows, cols], ref, "dp4a prefill9b up (sampled)")
    assert np.all(np.isfinite(y))
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(129, 19556, 544), (300, 20480, 1056), (129, 32768, 544),
                                   (300, 26000, 544)])
def test_tensor_path_stream_k(q8, M, N, K):
    """Shapes whose 128 x 256 tiles fill a partial last wave of the GPU: the tiles of that wave
    and one full wave are shared out as equal runs of scale windows, one per SM, and a run
    that splits a tile stores a partial that a second kernel adds.  (129, 19556): 154 tiles,
    the last, ragged column tile at both row tiles (one of them a single row); K = 544 is
    17 blocks, two windows of 16 and 1 blocks.  (129, 32768): 256 tiles, runs of 3.4 windows
    that touch up to three tiles.  (300, 26000): 306 tiles, runs over 154 of them followed by
    152 whole tiles.  Element by element, and deterministic."""
    rng = np.random.default_rng(M + N)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=True, outlier_frac=0.02)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    y_ref = O.linear(x, Wq_ref, Wd_ref, bf16=True)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    y = q8.q8_linear_ex(T(x), Wq, Wd, path="tensor")
    y2 = q8.q8_linear_ex(T(x), Wq, Wd, path="tensor")
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert_close(y.cpu().numpy(), y_ref, f"tensor stream-K M={M} N={N} K={K}")
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(1, 1000, 544), (77, 1000, 544), (128, 4096, 4096),
                                   (128, 19556, 1056), (100, 300, 512)])
def test_tensor_path_int8_weights(q8, M, N, K):
    """Up to 128 tokens the tensor path's GEMM reads the int8 weight codes by TMA and widens
    them to binary16 in shared memory itself (no separate widening pass): the results are
    the bits of the binary16 path on the same codes (the prepared-weights entry point) and
    match the oracle.  Ragged N, K of 17 and 33 blocks (a last stage with one block), and
    uniform split-K along K (4096 x 4096 and 19556 x 1056 at M = 128: 16 and 77 tiles)."""
    rng = np.random.default_rng(M * 7 + N + K)
    W = workloads.weights(rng, N, K)
    x, _ = workloads.activations(rng, M, K, bf16=True, outlier_frac=0.02)
    Wq_ref, Wd_ref = O.quantize_weights(W)
    y_ref = O.linear(x, Wq_ref, Wd_ref, bf16=True)
    Wq, Wd = q8.q8_quantize_weights(T(W))
    xt = T(x)
    y = q8.q8_linear_ex(xt, Wq, Wd, path="tensor")
    yp = q8.q8_linear_prepared(xt, q8.q8_weights_to_f16(Wq), Wd)
    torch.cuda.synchronize()
    assert torch.equal(y, yp)
    assert_close(y.cpu().numpy(), y_ref, f"tensor int8 weights M={M} N={N} K={K}")
    assert q8.q8_device_error() == 0
