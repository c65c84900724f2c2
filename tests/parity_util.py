"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""

import numpy as np
import torch

TOL = {"bf16": 1e-2, "f32": 1e-4}


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def relerr(got, ref, floor=0.0):
    """max|got - ref| / max(max|ref|, floor) over all compared elements."""
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    if not np.isfinite(g).all():
        return float("inf")
    den = max(float(np.abs(r).max()) if r.size else 0.0, floor, 1e-30)
    return float(np.abs(g - r).max() / den) if r.size else 0.0


def sample_rows(n, count, seed):
    """Sorted distinct row indices: the first and last 8 rows plus `count`
    seeded random rows (all rows when n is small)."""
    if n <= count + 16:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(8, n - 8), size=count, replace=False)
    return np.unique(np.concatenate([np.arange(8), mid, np.arange(n - 8, n)]))
