"""Parity of block-sparse causal attention (q8_bsa_attention) with the binary64 oracle.

Tolerance, from the arithmetic: scores are exact bf16 products summed in binary32
(relative ~1e-7) and the softmax runs in binary32, but the weights enter the P.V product
rounded to bfloat16 (at most 2^-9 relative each, while the row sum uses the unrounded
weights).  Averaged over the visible keys that is ~2e-3 relative on o: the bound is
relative-Frobenius <= 4e-3 and max-abs <= 1e-2 * max|o_ref| (both doubled for a bfloat16 o,
which adds one more rounding).
"""
import numpy as np
import pytest

import workloads
from oracle import bsa as OB
from tests.gpu_util import dev_tensor

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FRO, MAX = 4e-3, 1e-2


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


def _close(o, ref, what, k=1.0):
    o = np.asarray(o, np.float64)
    ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(o - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.max(np.abs(o - ref)) / max(np.max(np.abs(ref)), 1e-30)
    assert fro <= k * FRO and mx <= k * MAX, f"{what}: rel-Frobenius {fro:.2e}, max-abs {mx:.2e}"


def _run(q8, q, k, v, rp, ci, dtype=torch.float32):
    return q8.q8_bsa_attention(T(q), T(k), T(v), T(rp), T(ci), out_dtype=dtype)


@pytest.mark.parametrize("H,Hkv,Tn,density", [(4, 2, 256, 0.3), (2, 2, 64, 0.0), (8, 1, 512, 0.2),
                                               (3, 3, 192, 1.0), (16, 4, 1024, 0.1)])
def test_matches_the_oracle(q8, H, Hkv, Tn, density):
    rng = np.random.default_rng(H * Tn)
    q, k, v = workloads.bsa_qkv(rng, H, Hkv, Tn)
    rp, ci = workloads.bsa_mask(rng, H, Tn, density)
    ref = OB.attention(q, k, v, rp, ci)
    o = _run(q8, q, k, v, rp, ci).cpu().numpy()
    _close(o, ref, f"H={H} T={Tn}")
    o16 = _run(q8, q, k, v, rp, ci, torch.bfloat16).float().cpu().numpy()
    _close(o16, ref, f"H={H} T={Tn} bf16", k=2.0)
    o2 = _run(q8, q, k, v, rp, ci).cpu().numpy()
    assert np.array_equal(o, o2)                       # deterministic
    assert q8.q8_device_error() == 0


def test_dense_causal_and_scaled_queries(q8):
    rng = np.random.default_rng(7)
    q, k, v = workloads.bsa_qkv(rng, 2, 1, 256)
    q = workloads.bf16_bits_from_f32(workloads.f32_from_bf16_bits(q) * np.float32(4.0))  # peaky
    rp, ci = workloads.dense_causal_mask(2, 256)
    _close(_run(q8, q, k, v, rp, ci).cpu().numpy(), OB.attention(q, k, v, rp, ci), "dense, sharp")


@pytest.mark.parametrize("mask", ["dense", "sparse"])
def test_running_max_rising_across_blocks(q8, mask):
    """Keys scaled up block by block (3 + 3 kb, and random factors up to 24): each new block
    raises a row's maximum score by more than 2^8 in base 2 on most blocks, so the kernel
    moves its exponent reference and rescales O in the middle of the sweep; a row whose
    maximum stays within 2^8 keeps its reference."""
    rng = np.random.default_rng(21)
    H, Hkv, Tn = 4, 2, 512
    q, k, v = workloads.bsa_qkv(rng, H, Hkv, Tn)
    nb = Tn // 64
    kf = workloads.f32_from_bf16_bits(k).reshape(Hkv, nb, 64, 128)
    if mask == "dense":
        grow = (3.0 + 3.0 * np.arange(nb, dtype=np.float32))[None, :, None, None]
        rp, ci = workloads.dense_causal_mask(H, Tn)
    else:
        grow = rng.uniform(0.5, 24.0, (Hkv, nb, 1, 1)).astype(np.float32)
        rp, ci = workloads.bsa_mask(rng, H, Tn, 0.5)
    k = workloads.bf16_bits_from_f32((kf * grow).reshape(Hkv, Tn, 128))
    ref = OB.attention(q, k, v, rp, ci)
    _close(_run(q8, q, k, v, rp, ci).cpu().numpy(), ref, f"rising maxima, {mask}")
    _close(_run(q8, q, k, v, rp, ci, torch.bfloat16).float().cpu().numpy(), ref,
           f"rising maxima, {mask}, bf16", k=2.0)
    assert q8.q8_device_error() == 0


def test_empty_rows_and_bad_blocks(q8):
    rng = np.random.default_rng(8)
    H, Tn = 2, 256
    q, k, v = workloads.bsa_qkv(rng, H, H, Tn)
    nb = Tn // 64
    # head 0: query block 2 lists nothing; head 1: query block 1 lists block 3 (in the future)
    rows = {(0, 2): [], (1, 1): [0, 3]}
    row_ptr, cols = [0], []
    for h in range(H):
        for qb in range(nb):
            cols.extend(rows.get((h, qb), list(range(qb + 1))))
            row_ptr.append(len(cols))
    rp, ci = np.array(row_ptr, np.int32), np.array(cols, np.int32)
    o = _run(q8, q, k, v, rp, ci).cpu().numpy()
    assert not np.any(o[0, 128:192])                   # no visible key: zero
    assert q8.q8_device_error() & 256                  # the future block was flagged
    rows[(1, 1)] = [0]                                 # ... and skipped
    row_ptr, cols = [0], []
    for h in range(H):
        for qb in range(nb):
            cols.extend(rows.get((h, qb), list(range(qb + 1))))
            row_ptr.append(len(cols))
    ref = OB.attention(q, k, v, np.array(row_ptr, np.int32), np.array(cols, np.int32))
    _close(o, ref, "empty rows and a skipped block")
    assert q8.q8_device_error() == 0


def test_many_items_per_cta_with_empty_lists(q8):
    """1024 (head, query block) items, more than the kernel's CTAs, so each CTA walks several
    of them with two Q buffers in turn.  Empty block lists sit mid-walk (every fifth item of
    head 1) and at the walk's end (the lowest query blocks of the last key/value group, which
    the kernel takes last); their rows must be 0 and the others must match the oracle."""
    rng = np.random.default_rng(31)
    H, Hkv, Tn = 8, 2, 8192
    nb = Tn // 64
    q, k, v = workloads.bsa_qkv(rng, H, Hkv, Tn)
    rp0, ci0 = workloads.bsa_mask(rng, H, Tn, 0.1)
    empty = set()
    for qb in range(0, nb, 5):
        empty.add((1, qb))
    for h in range(H - H // Hkv, H):
        for qb in range(12):
            empty.add((h, qb))
    row_ptr, cols = [0], []
    for h in range(H):
        for qb in range(nb):
            r = h * nb + qb
            if (h, qb) not in empty:
                cols.extend(ci0[rp0[r]:rp0[r + 1]].tolist())
            row_ptr.append(len(cols))
    rp, ci = np.array(row_ptr, np.int32), np.array(cols, np.int32)
    o = _run(q8, q, k, v, rp, ci)
    o_np = o.cpu().numpy()
    for (h, qb) in empty:
        assert not np.any(o_np[h, 64 * qb:64 * qb + 64]), (h, qb)
    heads = np.concatenate([[0, H - 1, 1], rng.integers(0, H, 400)])
    toks = np.concatenate([[Tn - 1, 64 * 12, 64 * 5 + 3], rng.integers(0, Tn, 400)])
    keep = np.array([(int(h), int(t) // 64) not in empty for h, t in zip(heads, toks)])
    heads, toks = heads[keep], toks[keep]
    ref = OB.attention_at(q, k, v, rp, ci, heads, toks)
    _close(o_np[heads, toks], ref, "many items per CTA")
    assert np.array_equal(o_np, _run(q8, q, k, v, rp, ci).cpu().numpy())  # deterministic
    assert q8.q8_device_error() == 0


def test_binding_refuses_strided_block_lists(q8):
    """A strided int32 view of the block list would hand the kernel the wrong words: the
    binding refuses it before anything launches."""
    rng = np.random.default_rng(9)
    q, k, v = workloads.bsa_qkv(rng, 2, 2, 128)
    rp, ci = workloads.dense_causal_mask(2, 128)
    strided = T(np.repeat(ci, 2))[::2]
    assert torch.equal(strided.cpu(), torch.from_numpy(ci)) and not strided.is_contiguous()
    with pytest.raises(ValueError, match="col_idx"):
        q8.q8_bsa_attention(T(q), T(k), T(v), T(rp), strided)
    o = q8.q8_bsa_attention(T(q), T(k), T(v), T(rp), strided.contiguous())
    _close(o.cpu().numpy(), OB.attention(q, k, v, rp, ci), "contiguous copy")


def test_full_size_32k(q8):
    """32 query heads over 8 key/value heads, 32768 tokens, ~10 % of the causal blocks:
    sampled queries (the first and last of the sequence included) against the oracle."""
    cfg = workloads.BSA_32K
    rng = np.random.default_rng(9)
    q, k, v = workloads.bsa_qkv(rng, cfg["H"], cfg["Hkv"], cfg["T"], cfg["d"])
    rp, ci = workloads.bsa_mask(rng, cfg["H"], cfg["T"], cfg["density"])
    o = _run(q8, q, k, v, rp, ci)
    heads = np.concatenate([[0, cfg["H"] - 1], rng.integers(0, cfg["H"], 300)])
    toks = np.concatenate([[0, cfg["T"] - 1], rng.integers(0, cfg["T"], 300)])
    ref = OB.attention_at(q, k, v, rp, ci, heads, toks)
    got = o[torch.from_numpy(heads).cuda(), torch.from_numpy(toks).cuda()].cpu().numpy()
    _close(got, ref, "32K sampled")
    assert torch.isfinite(o).all()
    assert q8.q8_device_error() == 0
