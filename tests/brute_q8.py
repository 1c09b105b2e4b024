"""A second, deliberately naive Q8_0 implementation in pure Python, written apart from
the C oracle, used only to cross-check it on small inputs.

It uses Python integers for block sums, numpy binary32 scalars for the one division the
definition makes, numpy's own binary16 conversion for weight scales, and exact rational
arithmetic (fractions.Fraction) for the output sum, rounded once to binary32.
"""
import math
from fractions import Fraction

import numpy as np

QK = 32


def round_half_away(t: float) -> int:
    """Nearest integer, ties away from zero.  t holds a binary32 value exactly, so
    |t| + 0.5 is exact in binary64 and floor() decides correctly."""
    a = math.floor(abs(t) + 0.5)
    return a if t >= 0 else -a


def quant_block(vals):
    """vals: 32 binary32 values -> (codes list, binary32 scale as float)."""
    amax = np.float32(0.0)
    for v in vals:
        a = np.float32(abs(np.float32(v)))
        if a > amax:
            amax = a
    d = np.float32(amax / np.float32(127.0))
    if d == 0:
        return [0] * QK, 0.0
    codes = []
    for v in vals:
        c = round_half_away(float(np.float32(v) / d))
        codes.append(max(-127, min(127, c)))
    return codes, float(d)


def quant_rows(X):
    """X: 2-D float32 array -> (codes [rows][K], scales [rows][K/32])."""
    codes, scales = [], []
    for row in X:
        rc, rs = [], []
        for b in range(len(row) // QK):
            c, d = quant_block([float(v) for v in row[b * QK:(b + 1) * QK]])
            rc.extend(c)
            rs.append(d)
        codes.append(rc)
        scales.append(rs)
    return codes, scales


def f16_bits(d: float) -> int:
    return int(np.array([d], dtype=np.float32).astype(np.float16).view(np.uint16)[0])


def f16_value(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0])


def block_sum(a, b, blk):
    return sum(a[blk * QK + j] * b[blk * QK + j] for j in range(QK))


def linear_exact(xc, xs, wc, wbits):
    """Exact rational y, rounded once to binary32."""
    M, N = len(xc), len(wc)
    nb = len(xs[0])
    y = np.zeros((M, N), np.float32)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for blk in range(nb):
                s = block_sum(xc[m], wc[n], blk)
                acc += Fraction(f16_value(wbits[n][blk])) * Fraction(xs[m][blk]) * s
            y[m, n] = np.float32(float(acc)) if acc == 0 else np.float32(_round_f32(acc))
    return y


def _round_f32(q: Fraction) -> float:
    """Round an exact rational to the nearest binary32 (ties to even)."""
    f = float(q)  # nearest binary64 (correctly rounded by Fraction.__float__)
    c = np.float32(f)
    # A double rounding (rational -> binary64 -> binary32) can only go wrong when the
    # binary64 value sits exactly on a binary32 midpoint; settle that case exactly.
    lo = np.nextafter(c, np.float32(-np.inf))
    hi = np.nextafter(c, np.float32(np.inf))
    best = c
    for cand in (lo, hi):
        if abs(Fraction(float(cand)) - q) < abs(Fraction(float(best)) - q):
            best = cand
    return float(best)
