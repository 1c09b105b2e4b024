"""Helpers for the GPU parity tests: moving seeded inputs to the device, and the
tolerance for binary32 outputs.

Tolerance (the order of the binary32 sum is not fixed, codes/scales/block sums are exact):
relative Frobenius error <= 1e-5 and max |y - y_ref| <= 1e-4 * max |y_ref|.  The GPU sums
about K/32 rescaled block terms in binary32 (relative error ~ sqrt(K/32) * 2^-24 ~ 1e-6 at
K = 17408), so the bound has an order of magnitude of headroom.
"""
import numpy as np

REL_FRO = 1e-5
REL_MAX = 1e-4


def dev_tensor(a, torch, device="cuda"):
    """numpy -> CUDA tensor; uint16 arrays are bfloat16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def close(y, ref):
    """(ok, relative Frobenius error, max abs error / max |ref|)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        ok = bool(np.all(y == ref))
        return ok, 0.0 if ok else np.inf, 0.0 if ok else np.inf
    fro = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    mx = np.max(np.abs(y - ref)) / scale
    return bool(fro <= REL_FRO and mx <= REL_MAX), float(fro), float(mx)


def assert_close(y, ref, what=""):
    ok, fro, mx = close(y, ref)
    assert ok, f"{what}: rel-Frobenius {fro:.3e} (<= {REL_FRO}), max-abs/max|ref| {mx:.3e} (<= {REL_MAX})"


def sample_indices(rng, M, N, count):
    """Sampled (row, col) pairs covering the corners, the first/last row and column, and
    random interior points."""
    rows = [0, 0, M - 1, M - 1] + list(rng.integers(0, M, count))
    cols = [0, N - 1, 0, N - 1] + list(rng.integers(0, N, count))
    edge = min(64, N)
    rows += [0] * edge + [M - 1] * edge
    cols += list(range(N - edge, N)) + list(range(edge))
    return np.array(rows, np.int64), np.array(cols, np.int64)
