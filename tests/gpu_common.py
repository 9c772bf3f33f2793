"""Shared helpers for the GPU parity tests: the tolerances and the comparison.

Tolerances (fixed by the specification of the path):
* attention / decode output O (bf16): max |O - O*| <= 2e-2 and mean |O - O*| <= 2e-3
* LSE (fp32): max |LSE - LSE*| <= 1e-3
* RMSNorm output (bf16): |y - y*| <= 1e-2 |y*| + 1e-6 element-wise
where * marks the float64 oracle evaluated on the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
NORM_REL = 1e-2
NORM_ABS_FLOOR = 1e-6


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from exact_tiled_attention_attn_gb300.build import build
    build()
    import exact_tiled_attention_attn_gb300 as attn
    attn.lib()
    return attn


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_round(v):
    """Round-to-nearest-even to bf16 of float64 values (8 significant bits), from frexp."""
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def assert_attn_close(o, lse, O, L, what=""):
    o = f64(o) if isinstance(o, torch.Tensor) else o
    err = np.abs(o - O)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert err.max() <= O_MAX_ABS, f"{what}: max |O - O*| = {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean |O - O*| = {err.mean():.3e}"
    if lse is not None:
        l = f64(lse) if isinstance(lse, torch.Tensor) else lse
        e2 = np.abs(l - L)
        assert e2.max() <= LSE_MAX_ABS, f"{what}: max |LSE - LSE*| = {e2.max():.3e}"
    return float(err.max()), float(err.mean())


def assert_norm_close(y, Y, what=""):
    y = f64(y) if isinstance(y, torch.Tensor) else y
    bad = np.abs(y - Y) > NORM_REL * np.abs(Y) + NORM_ABS_FLOOR
    assert not bad.any(), f"{what}: {bad.sum()} elements outside 1e-2 relative, worst " \
                          f"{(np.abs(y - Y) / (np.abs(Y) + NORM_ABS_FLOOR)).max():.3e}"
