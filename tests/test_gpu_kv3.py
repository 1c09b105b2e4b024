"""Parity of the 3-bit KV-cache codec (q8_kv3_encode / q8_kv3_decode) with the oracle.

Bit-exact: the codes and scales of the encoder (the rotation, the pairwise sum of squares
and every decision are the same binary32 operations in the same order on both sides), the
binary32 output of the decoder, and the bfloat16 output (round to nearest even of the
binary32 one).
"""
import numpy as np
import pytest

import workloads
from oracle import kv3 as OK
from tests.gpu_util import dev_tensor

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


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _crafted(rng):
    """Zero groups, exact-zero rotations, unit vectors, large and small groups (inside the
    binary32 range of the sum of squares), a group whose sum of squares underflows, and a
    group with a negative-zero rotation output."""
    g = []
    g.append(np.zeros(128, np.float32))
    e = np.zeros(128, np.float32)
    e[0] = e[1] = 1.0
    g.append(e)
    for j, c in ((0, 1.0), (37, -0.5), (127, 8.0)):
        u = np.zeros(128, np.float32)
        u[j] = c
        g.append(u)
    g.append(rng.standard_normal(128).astype(np.float32) * np.float32(1e15))
    g.append(rng.standard_normal(128).astype(np.float32) * np.float32(1e-15))
    g.append(rng.standard_normal(128).astype(np.float32) * np.float32(1e-30))  # s underflows to 0
    g.append(np.full(128, 3.0, np.float32))
    z = np.zeros(128, np.float32)  # rotation output 127 is -0 while s != 0: a positive code
    z[0] = -0.0
    z[2] = z[3] = 5.0
    g.append(z)
    return np.stack(g)


@pytest.mark.parametrize("n,bf16", [(1, True), (9, False), (1000, True), (4097, False), (33333, True)])
def test_encode_decode_bit_exact(q8, n, bf16):
    rng = np.random.default_rng(n)
    x = workloads.kv_groups(rng, n, 1, 128, outlier_frac=0.03, bf16=bf16)
    if not bf16:
        cr = _crafted(rng)
        k = min(n, len(cr))
        x[:k] = cr[:k]
    words, scales = OK.encode(x, bf16=bf16)
    c, s = q8.q8_kv3_encode(T(x))
    assert np.array_equal(_u32(c), words)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    ref = OK.decode(words, scales)
    out32 = q8.q8_kv3_decode(c, s, torch.float32).cpu().numpy()
    assert np.array_equal(out32.view(np.uint32), ref.view(np.uint32))
    out16 = q8.q8_kv3_decode(c, s, torch.bfloat16)
    want16 = torch.from_numpy(ref).to(torch.bfloat16)
    assert torch.equal(out16.cpu().view(torch.int16), want16.view(torch.int16))
    assert q8.q8_device_error() == 0


def test_decode_of_oracle_codes(q8):
    """The decoder on codes it did not produce: every 3-bit value at every position."""
    rng = np.random.default_rng(9)
    n = 513
    words = rng.integers(0, 2 ** 32, (n, 12), dtype=np.uint64).astype(np.uint32)
    scales = (rng.random(n) * 10).astype(np.float32)
    scales[0] = 0.0
    ref = OK.decode(words, scales)
    out = q8.q8_kv3_decode(T(words.view(np.int32)), T(scales), torch.float32).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


def test_outputs_stay_inside_their_buffers(q8):
    rng = np.random.default_rng(10)
    n = 77
    x = workloads.kv_groups(rng, n, 1, 128)
    pad = 64
    cbig = torch.full((n * 12 + 2 * pad,), -1, dtype=torch.int32, device="cuda")
    sbig = torch.full((n + 2 * pad,), float("nan"), device="cuda")
    c = cbig[pad:pad + n * 12].view(n, 12)
    s = sbig[pad:pad + n]
    q8.q8_kv3_encode(T(x), codes=c, scales=s)
    obig = torch.full((n * 128 + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = obig[pad:pad + n * 128].view(n, 128)
    q8.q8_kv3_decode(c, s, torch.bfloat16, out=o)
    torch.cuda.synchronize()
    assert (cbig[:pad] == -1).all() and (cbig[pad + n * 12:] == -1).all()
    assert torch.isnan(sbig[:pad]).all() and torch.isnan(sbig[pad + n:]).all()
    assert torch.isnan(obig[:pad]).all() and torch.isnan(obig[pad + n * 128:]).all()
    assert torch.isfinite(o).all()


def test_empty(q8):
    c, s = q8.q8_kv3_encode(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"))
    assert c.shape == (0, 12)
    assert q8.q8_kv3_decode(c, s).shape == (0, 128)


def test_full_size_256k_context_layer(q8):
    """One attention layer's keys at a 256K-token context (262144 tokens x 4 heads x 256
    channels = 2,097,152 groups): sampled groups against the oracle, and the whole cache's
    round-trip distortion."""
    rng = np.random.default_rng(11)
    x = workloads.kv_groups(rng, **workloads.KV3_LAYER_256K)
    xt = T(x)
    c, s = q8.q8_kv3_encode(xt)
    n = x.shape[0]
    idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 3000)]))
    words, scales = OK.encode(x[idx], bf16=True)
    assert np.array_equal(_u32(c[torch.from_numpy(idx).cuda()]), words)
    assert np.array_equal(s[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint32), scales.view(np.uint32))
    y = q8.q8_kv3_decode(c, s, torch.float32)
    ref = OK.decode(words, scales)
    assert np.array_equal(y[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint32), ref.view(np.uint32))
    xf = xt.float()
    rel = float(((xf - y) ** 2).sum() / (xf ** 2).sum())
    assert 0.02 < rel < 0.05, rel
    assert q8.q8_device_error() == 0
