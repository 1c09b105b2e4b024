"""Seeded synthetic inputs for the Q8_0 linear layer (shared by tests and the benchmark).

This module only draws random numbers and shapes them; it holds none of the method's
arithmetic (no quantization, no scales, no dot products), so it can feed both the CUDA
library and the CPU oracle without coupling them.

Recipe (numpy PCG64 via default_rng):
  * weights  W = standard_normal((N, K), float32) * 0.02
  * activations x = standard_normal((M, K), float32); for the outlier workload a fixed
    set of round(0.01*K) channels (K indices, the same for every row) is multiplied by
    20 in float32; then x is rounded to bfloat16 (nearest-even) unless the workload is
    float32.
  * one generator per (workload, projection) for weights, and one per (workload,
    projection, M) for activations, seeded as listed in SEEDS below.
  * KV-cache groups (the 3-bit codec): keys or values of `tokens` tokens x `heads` heads
    x `head_dim` channels, standard_normal float32 times a per-channel gain that is 1
    except on round(outlier_frac * head_dim) channels (the same for every token and head)
    where it is `gain`; rounded to bfloat16; cut into 128-element groups (a 256-wide head
    is two groups).
  * block-sparse attention: q, k, v standard_normal float32 rounded to bfloat16; the block
    pattern per head and 64-token query block keeps the first key block, the two blocks
    ending at the diagonal, and each other earlier block with probability 0.1.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np

QK = 32


def bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return ((u >> 16) & 0xFFFF).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(rng: np.random.Generator, N: int, K: int, std: float = 0.02) -> np.ndarray:
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def activations(rng: np.random.Generator, M: int, K: int, bf16: bool = True,
                outlier_frac: float = 0.0, outlier_gain: float = 20.0):
    """Returns (x, outlier_channels): x is uint16 bf16 bits when bf16 else float32."""
    x = rng.standard_normal((M, K), dtype=np.float32)
    idx = np.zeros(0, np.int64)
    if outlier_frac > 0.0:
        cnt = int(round(outlier_frac * K))
        idx = np.sort(rng.choice(K, size=cnt, replace=False)).astype(np.int64)
        x[:, idx] *= np.float32(outlier_gain)
    if bf16:
        return bf16_bits_from_f32(x), idx
    return x, idx


@dataclass
class Linear:
    """One projection shape: y[M,N] = x[M,K] . W[N,K]^T."""
    name: str
    K: int
    N: int


@dataclass
class Workload:
    name: str
    seed: int
    projections: List[Linear]
    Ms: List[int]
    bf16: bool = True
    outlier_frac: float = 0.0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def weight_rng(self, p: int) -> np.random.Generator:
        return np.random.default_rng([self.seed, 1000 + p])

    def act_rng(self, p: int, mi: int) -> np.random.Generator:
        return np.random.default_rng([self.seed, 2000 + 100 * mi + p])

    def make_weights(self, p: int) -> np.ndarray:
        pr = self.projections[p]
        return weights(self.weight_rng(p), pr.N, pr.K)

    def make_act(self, p: int, mi: int):
        pr = self.projections[p]
        return activations(self.act_rng(p, mi), self.Ms[mi], pr.K, bf16=self.bf16,
                           outlier_frac=self.outlier_frac)

    def cases(self) -> List[Tuple[int, int]]:
        """(projection index, M index) pairs, M outermost."""
        return [(p, mi) for mi in range(len(self.Ms)) for p in range(len(self.projections))]


HIDDEN = 5120
FFN_27B = 17408

WORKLOADS = {
    # tiny Q8_0 linear, float32 activations
    "tiny": Workload("tiny", 0, [Linear("tiny", 512, 256)], [16], bf16=False),
    # decode: FFN up-projection of a dense ~9B-class layer, M = 1 and batched decode
    "decode": Workload("decode", 1, [Linear("up", 4096, 12288)], [1, 4, 16, 64]),
    # prefill, 9B-class up and down projections
    "prefill9b": Workload("prefill9b", 2, [Linear("up", 4096, 12288), Linear("down", 12288, 4096)],
                          [2048]),
    # prefill, 27B-class shapes, 1% of activation channels scaled x20
    "prefill27b": Workload("prefill27b", 3, [Linear("up", HIDDEN, FFN_27B),
                                             Linear("down", FFN_27B, HIDDEN)], [8192],
                           outlier_frac=0.01),
    # every linear of a synthetic hybrid layer with hidden size 5120
    "sweep": Workload("sweep", 4, [Linear("q", HIDDEN, HIDDEN), Linear("k", HIDDEN, HIDDEN),
                                   Linear("v", HIDDEN, HIDDEN), Linear("o", HIDDEN, HIDDEN),
                                   Linear("gate", HIDDEN, FFN_27B), Linear("up", HIDDEN, FFN_27B),
                                   Linear("down", FFN_27B, HIDDEN),
                                   Linear("gdn_in", HIDDEN, 10240)],
                      [1, 4, 16, 128, 512, 2048, 8192]),
}


def algorithmic_bytes(M: int, N: int, K: int, x_bytes: int = 2) -> int:
    """Bytes a Q8_0 linear must move at least once: codes + binary16 scales of W,
    the activations, and the float32 output."""
    return N * K + 2 * N * (K // QK) + x_bytes * M * K + 4 * M * N


def algorithmic_ops(M: int, N: int, K: int) -> int:
    """int8-equivalent multiply-add operations (2 per MAC); block rescales excluded."""
    return 2 * M * N * K


KV3_GROUP = 128


def kv_groups(rng: np.random.Generator, tokens: int, heads: int, head_dim: int = 256,
              outlier_frac: float = 0.02, gain: float = 10.0, bf16: bool = True) -> np.ndarray:
    """Synthetic keys or values as [tokens * heads * head_dim / 128, 128] groups
    (bfloat16 bits as uint16, or float32)."""
    x = rng.standard_normal((tokens, heads, head_dim), dtype=np.float32)
    cnt = int(round(outlier_frac * head_dim))
    if cnt:
        idx = rng.choice(head_dim, size=cnt, replace=False)
        x[:, :, idx] *= np.float32(gain)
    x = x.reshape(-1, KV3_GROUP)
    return bf16_bits_from_f32(x) if bf16 else x


# 256K-token context of the post's 3-bit KV cache: one attention layer's keys (or values),
# 4 KV heads of 256 channels
KV3_LAYER_256K = dict(tokens=262144, heads=4, head_dim=256)


BSA_BLOCK = 64


def bsa_qkv(rng: np.random.Generator, H: int, Hkv: int, T: int, d: int = 128):
    """Synthetic queries, keys and values: standard_normal float32 rounded to bfloat16 bits,
    q [H,T,d], k and v [Hkv,T,d]."""
    q = bf16_bits_from_f32(rng.standard_normal((H, T, d), dtype=np.float32))
    k = bf16_bits_from_f32(rng.standard_normal((Hkv, T, d), dtype=np.float32))
    v = bf16_bits_from_f32(rng.standard_normal((Hkv, T, d), dtype=np.float32))
    return q, k, v


def bsa_mask(rng: np.random.Generator, H: int, T: int, density: float = 0.1, local: int = 2):
    """A block-sparse causal pattern as CSR (row_ptr [H*nb+1], col_idx): per head and query
    block qb, the first key block (the attention sink), the `local` blocks ending at qb (the
    diagonal included), and each other earlier block with probability `density`."""
    nb = T // BSA_BLOCK
    row_ptr = [0]
    cols = []
    for _h in range(H):
        for qb in range(nb):
            keep = rng.random(qb + 1) < density
            keep[0] = True
            keep[max(0, qb - local + 1):qb + 1] = True
            sel = np.nonzero(keep)[0]
            cols.extend(sel.tolist())
            row_ptr.append(len(cols))
    return np.array(row_ptr, np.int32), np.array(cols, np.int32)


def dense_causal_mask(H: int, T: int):
    """Every block at or below the diagonal: plain causal attention."""
    nb = T // BSA_BLOCK
    row_ptr = [0]
    cols = []
    for _h in range(H):
        for qb in range(nb):
            cols.extend(range(qb + 1))
            row_ptr.append(len(cols))
    return np.array(row_ptr, np.int32), np.array(cols, np.int32)


# long prefill with block-sparse attention: 32 query heads over 8 key/value heads, head
# dim 128, 32768 tokens, about 10 % of the causal key blocks
BSA_32K = dict(H=32, Hkv=8, T=32768, d=128, density=0.1)
