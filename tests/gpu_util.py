"""Helpers for the GPU parity tests: device transfer and oracle comparison."""

import numpy as np
import torch

from oracle import nvfp4_oracle as O


def dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_within(got, ref, abs_sum, alpha, what=""):
    """Elementwise |got - ref| <= 2^-8 |ref| + 1e-6 |alpha| sum|a b|, and finite."""
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    tol = O.tolerance(ref, abs_sum, alpha)
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; max err/tol = "
            f"{float(np.max(err / np.maximum(tol, 1e-300))):.3g}; first {idx.tolist()}; "
            f"got {got[bad][:4]} ref {ref[bad][:4]}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def sample_points(M, N, n, seed=1234):
    g = np.random.default_rng(seed)
    return g.integers(0, M, n), g.integers(0, N, n)


def corner_tiles(M, N, t=128):
    """The four corner t x t tiles (row0, row1, col0, col1) of an M x N output."""
    r_last = max(0, M - t)
    c_last = max(0, N - t)
    out = []
    for r0 in sorted({0, r_last}):
        for c0 in sorted({0, c_last}):
            out.append((r0, min(M, r0 + t), c0, min(N, c0 + t)))
    return out
