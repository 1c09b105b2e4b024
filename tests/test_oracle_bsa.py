"""Pins of the block-sparse attention oracle (oracle/bsa_oracle.c) to facts that do not come
from the oracle itself.

- equal value rows come back unchanged (the weights sum to one);
- zero keys give the plain mean of the visible value rows (visibility written out here
  from the block lists and causality);
- the first query of the sequence sees only itself: its own value row, through the
  grouped-query head mapping;
- a two-key closed form fixes the softmax and its 1/sqrt(d) scale;
- a sharp softmax (queries scaled by 64) returns the value row of the best visible key;
- masked blocks and future tokens are invisible; heads sharing a key/value head agree;
- against a library routine: PyTorch's scaled_dot_product_attention in binary64 on the
  CPU, plain causal for the dense mask and with the block-and-causal visibility written out
  as an explicit boolean mask for a sparse one.
"""
import math

import numpy as np
import pytest

import workloads
from oracle import bsa

B = 64


def _f(bits):
    return workloads.f32_from_bf16_bits(bits).astype(np.float64)


def _visible(row_ptr, col_idx, h, t, T):
    nb = T // B
    qb = t // B
    keys = []
    for e in range(row_ptr[h * nb + qb], row_ptr[h * nb + qb + 1]):
        kb = col_idx[e]
        keys.extend(j for j in range(kb * B, (kb + 1) * B) if j <= t)
    return keys


def _case(seed, H=4, Hkv=2, T=256, d=128, density=0.3):
    rng = np.random.default_rng(seed)
    q, k, v = workloads.bsa_qkv(rng, H, Hkv, T, d)
    rp, ci = workloads.bsa_mask(rng, H, T, density)
    return q, k, v, rp, ci


def test_equal_value_rows_come_back():
    q, k, v, rp, ci = _case(1)
    v[:] = v[0, 0]
    o = bsa.attention(q, k, v, rp, ci)
    assert np.array_equal(o, np.broadcast_to(_f(v[0, 0]).astype(np.float32), o.shape))


def test_zero_keys_average_the_visible_values():
    q, k, v, rp, ci = _case(2)
    k[:] = 0
    o = bsa.attention(q, k, v, rp, ci)
    H, T, _ = q.shape
    group = H // k.shape[0]
    vf = _f(v)
    for h in range(H):
        for t in range(0, T, 7):
            keys = _visible(rp, ci, h, t, T)
            want = vf[h // group, keys].mean(axis=0)
            assert np.allclose(o[h, t], want, rtol=1e-6, atol=1e-7), (h, t)


def test_first_query_sees_only_itself():
    q, k, v, rp, ci = _case(3, H=8, Hkv=2)
    o = bsa.attention(q, k, v, rp, ci)
    for h in range(8):
        assert np.array_equal(o[h, 0], _f(v[h // 4, 0]).astype(np.float32)), h


def test_two_key_closed_form_fixes_the_scale():
    H, Hkv, T, d = 1, 1, 64, 128
    q = np.zeros((H, T, d), np.float32)
    k = np.zeros((Hkv, T, d), np.float32)
    v = np.zeros((Hkv, T, d), np.float32)
    q[0, 1, :4] = 1.0                      # query 1 sees keys 0 and 1
    k[0, 0, :4] = 0.5                      # q.k0 = 2
    k[0, 1, :4] = 3.0                      # q.k1 = 12
    v[0, 0, 0] = 1.0
    v[0, 1, 1] = 1.0
    bits = [workloads.bf16_bits_from_f32(a) for a in (q, k, v)]
    rp, ci = workloads.dense_causal_mask(H, T)
    o = bsa.attention(*bits, rp, ci)
    r = math.exp((12.0 - 2.0) / math.sqrt(d))
    assert o[0, 1, 0] == pytest.approx(1.0 / (1.0 + r), rel=1e-7)
    assert o[0, 1, 1] == pytest.approx(r / (1.0 + r), rel=1e-7)


def test_sharp_softmax_picks_the_best_key():
    q, k, v, rp, ci = _case(4, H=2, Hkv=1, T=192)
    q = workloads.bf16_bits_from_f32(workloads.f32_from_bf16_bits(q) * np.float32(64.0))
    o = bsa.attention(q, k, v, rp, ci)
    qf, kf, vf = _f(q), _f(k), _f(v)
    checked = 0
    for h in range(2):
        for t in range(0, 192, 5):
            keys = _visible(rp, ci, h, t, 192)
            s = kf[0, keys] @ qf[h, t]
            best = keys[int(np.argmax(s))]
            if np.sort(s)[-1] - (np.sort(s)[-2] if len(s) > 1 else -np.inf) > 200:
                assert np.allclose(o[h, t], vf[0, best], atol=1e-6), (h, t)
                checked += 1
    assert checked > 20


def test_masked_blocks_and_future_tokens_are_invisible():
    q, k, v, rp, ci = _case(5, H=2, Hkv=1, T=256)
    o = bsa.attention(q, k, v, rp, ci)
    nb = 4
    for h in range(2):
        for qb in range(nb):
            active = set(ci[rp[h * nb + qb]:rp[h * nb + qb + 1]].tolist())
            hidden = [kb for kb in range(qb) if kb not in active]
            if not hidden:
                continue
            k2, v2 = k.copy(), v.copy()
            for kb in hidden:
                k2[:, kb * B:(kb + 1) * B] ^= np.uint16(0x1234)
                v2[:, kb * B:(kb + 1) * B] ^= np.uint16(0x0F0F)
            o2 = bsa.attention(q, k2, v2, rp, ci)
            assert np.array_equal(o2[h, qb * B:(qb + 1) * B], o[h, qb * B:(qb + 1) * B])
    # token t + 1 and later never change o_t
    k3, v3 = k.copy(), v.copy()
    k3[:, 101:] ^= np.uint16(0x2222)
    v3[:, 101:] ^= np.uint16(0x2222)
    o3 = bsa.attention(q, k3, v3, rp, ci)
    assert np.array_equal(o3[:, :101], o[:, :101])
    assert not np.array_equal(o3[:, 101:], o[:, 101:])


def test_heads_sharing_a_kv_head_agree():
    q, k, v, rp, ci = _case(6, H=4, Hkv=2)
    q[1] = q[0]                         # heads 0 and 1 share kv head 0
    q[2] = q[0]                         # head 2 reads kv head 1
    rp1, ci1 = workloads.dense_causal_mask(4, 256)
    o = bsa.attention(q, k, v, rp1, ci1)
    assert np.array_equal(o[0], o[1])
    assert not np.array_equal(o[0], o[2])


def _visibility(row_ptr, col_idx, H, T):
    """[H, T, T] booleans: query t of head h sees key j (listed block, j <= t)."""
    nb = T // B
    m = np.zeros((H, T, T), bool)
    for h in range(H):
        for qb in range(nb):
            for kb in col_idx[row_ptr[h * nb + qb]:row_ptr[h * nb + qb + 1]]:
                m[h, qb * B:(qb + 1) * B, kb * B:(kb + 1) * B] = True
    return m & np.tril(np.ones((T, T), bool))


def _sdpa(q, k, v, mask=None):
    """torch's scaled_dot_product_attention in binary64 on the CPU (scale 1/sqrt(d)), each
    key/value head repeated for the query heads that share it."""
    torch = pytest.importorskip("torch")
    g = q.shape[0] // k.shape[0]
    tq = torch.from_numpy(_f(q))
    tk = torch.from_numpy(_f(k)).repeat_interleave(g, 0)
    tv = torch.from_numpy(_f(v)).repeat_interleave(g, 0)
    if mask is None:
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    else:
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask))
    return o.numpy()


def _agree(o, ref):
    # the oracle rounds a binary64 result once to binary32
    assert np.allclose(o, ref, rtol=2.0 ** -23, atol=1e-12 * np.max(np.abs(ref)))


def test_dense_causal_mask_is_library_causal_attention():
    q, k, v, _, _ = _case(10, H=4, Hkv=2, T=192)
    rp, ci = workloads.dense_causal_mask(4, 192)
    _agree(bsa.attention(q, k, v, rp, ci), _sdpa(q, k, v))


def test_block_sparse_is_library_attention_under_the_block_mask():
    q, k, v, rp, ci = _case(11, H=4, Hkv=2, T=512, density=0.3)
    mask = _visibility(rp, ci, 4, 512)
    assert mask.any(axis=2).all()          # every query sees itself: no empty softmax
    assert all(not np.array_equal(mask[0], mask[h]) for h in range(1, 4))   # per-head lists
    _agree(bsa.attention(q, k, v, rp, ci), _sdpa(q, k, v, mask))


def test_sampled_queries_equal_the_full_output():
    """attention_at (the sampled form the full-size GPU test uses) returns, bit for bit, the
    rows of the full output at the sampled (head, token) pairs."""
    q, k, v, rp, ci = _case(12, H=4, Hkv=2, T=256, density=0.3)
    o = bsa.attention(q, k, v, rp, ci)
    rng = np.random.default_rng(12)
    heads = rng.integers(0, 4, 40)
    toks = rng.integers(0, 256, 40)
    assert np.array_equal(bsa.attention_at(q, k, v, rp, ci, heads, toks), o[heads, toks])
