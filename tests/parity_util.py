"""Helpers for the GPU parity tests: host copies and bit comparisons.

The oracle runs on host copies of exactly the bytes the GPU consumed.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

CHUNK = 4096
TOL = 1e-6   # max-abs error normalised by max |reference|, for the mean and theta


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32 if a.dtype == np.float32 else np.uint8)


def assert_bit_equal(got: np.ndarray, ref: np.ndarray, what: str):
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    g, r = bits(got), bits(ref)
    if not np.array_equal(g, r):
        bad = np.flatnonzero((g != r).reshape(-1))
        raise AssertionError(f"{what}: {bad.size} of {g.size} differ, first at {bad[:8].tolist()}")


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, tol: float = TOL):
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max()) if ref.size else 0.0
    assert err <= tol * max(scale, np.finfo(np.float32).tiny), \
        f"{what}: max err {err:.3e} > {tol:g} x {scale:.3e}"
