"""Float64 oracle for RMSNorm.

TEST INFRASTRUCTURE ONLY (see the package docstring).

y[t, j] = x[t, j] / sqrt(mean_j x[t, j]^2 + eps) * w[j]; eps sits inside the
square root and the mean runs over the D axis of each row.
Source: "Module 07: Fused operators and FlashAttention", section "Fused
RMSNorm" (the formula) and section "Assignment 07.1: fused_rms_norm" (eps
under the root, mean over D, not over T).
"""
from __future__ import annotations

import numpy as np


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x: [T, D] float64, w: [D] float64 -> y [T, D] float64."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)[None, :]


def rmsnorm_rows(x: np.ndarray, w: np.ndarray, eps: float, rows) -> np.ndarray:
    """The same definition evaluated for selected rows only."""
    rows = np.asarray(rows, dtype=np.int64)
    return rmsnorm(np.asarray(x)[rows], w, eps)
