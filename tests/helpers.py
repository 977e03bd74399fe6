"""Comparison helpers shared by the GPU parity tests."""

import numpy as np

# Tolerances on max relative error: fp32 inputs 1e-4, bf16 inputs 2e-2 (fp32 accumulation).
TOL = {"f32": 1e-4, "bf16": 2e-2}


def max_rel_err(got, want):
    """max_e |got - want| / max(|want|, 1e-3 * max|want|): relative error with a floor
    so that near-zero reference elements do not dominate."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    if want.size == 0:
        return 0.0
    floor = 1e-3 * max(float(np.max(np.abs(want))), 1e-300)
    return float(np.max(np.abs(got - want) / np.maximum(np.abs(want), floor)))


def normwise_err(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if want.size == 0:
        return 0.0
    return float(np.max(np.abs(got - want)) / max(float(np.max(np.abs(want))), 1e-300))
