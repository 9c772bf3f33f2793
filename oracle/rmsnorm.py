"""Float64 oracle for RMSNorm.

TEST INFRASTRUCTURE ONLY (see the package docstring).

y[t, j] = x[t, j] / sqrt(mean_j x[t, j]^2 + eps) * w[j]; eps sits inside the
square root and the mean runs over the D axis of each row.
Source: "Module 07: Fused operators and FlashAttention", section "Fused
RMSNorm" (the formula) and section "Assignment 07.1: fused_rms_norm" (eps
under the root, mean over D, not over T).

The residual form (same module, the end of the RMSNorm assignment: the kernel
also folds in the residual add, rms_norm(x + residual), saving one more pass):
h = x + r (the new residual stream) and y = RMSNorm(h) * w, both from the exact
sum. How the GPU splits the row's sum of squares ("Chapter 5. Operators and
runtime", section 5.2.4) changes only the rounding, not this definition.
"""
from __future__ import annotations

import numpy as np


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x: [T, D] float64, w: [D] float64 -> y [T, D] float64."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)[None, :]


def rmsnorm_residual(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float):
    """x, r: [T, D], w: [D] -> (y, h): h = x + r, y = RMSNorm(h) * w (float64)."""
    h = np.asarray(x, dtype=np.float64) + np.asarray(r, dtype=np.float64)
    return rmsnorm(h, w, eps), h
