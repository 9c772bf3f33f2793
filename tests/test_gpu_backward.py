"""Parity of the backward pass (attn_bwd through the C ABI) with the float64 oracle.

The GPU backward takes the GPU forward's O (bf16) and LSE (fp32), as a training step
would; the oracle recomputes everything from the same bf16 inputs in float64. Tolerance
(derived from the arithmetic: P and dS are rounded to bf16 for the tensor-core
products, relative 2^-9, D_i comes from the bf16 O, and the outputs are rounded once
to bf16, relative 2^-9): for each of dQ, dK, dV, max |g - g*| <= 2e-2 max |g*| and
mean |g - g*| <= 1e-2 mean |g*|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import f64, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


def _grad_close(got, want, what):
    got = f64(got)
    err = np.abs(got - want)
    scale_max, scale_mean = np.abs(want).max(), np.abs(want).mean()
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max() <= 2e-2 * scale_max + 1e-6, f"{what}: max err {err.max():.3e} vs max |ref| {scale_max:.3e}"
    assert err.mean() <= 1e-2 * scale_mean + 1e-7, f"{what}: mean err {err.mean():.3e} vs mean |ref| {scale_mean:.3e}"
    return err.max() / max(scale_max, 1e-30)


def _case(attn, B, Hq, Hkv, Tq, Tk, d, causal, seed):
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed)
    do = W.grad_output(B, Hq, Tq, d, seed)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = attn.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    qf, kf, vf = f64(q), f64(k), f64(v)
    O, L = oracle.attention(qf, kf, vf, causal, scale)
    dQ, dK, dV = oracle.attention_backward(qf, kf, vf, O, L, f64(do), causal, scale)
    tag = f"B{B} Hq{Hq} Hkv{Hkv} Tq{Tq} Tk{Tk} d{d} causal{causal}"
    rel = [_grad_close(dq, dQ, "dQ " + tag), _grad_close(dk, dK, "dK " + tag), _grad_close(dv, dV, "dV " + tag)]
    print(tag, "max rel err dQ dK dV:", [f"{r:.2e}" for r in rel])
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (8, 2), (3, 1)])
def test_backward_grouping_modes(attn, d, causal, Hq, Hkv):
    _case(attn, 2, Hq, Hkv, 300, 300, d, causal, seed=1200 + Hq + d)


@pytest.mark.parametrize("T", [1, 127, 128, 129, 640])
def test_backward_lengths(attn, T):
    _case(attn, 1, 4, 2, T, T, 128, True, seed=1300 + T)


@pytest.mark.parametrize("Tq,Tk,causal", [(100, 300, False), (300, 100, False), (100, 300, True), (300, 100, True)])
def test_backward_rectangular(attn, Tq, Tk, causal):
    _case(attn, 1, 2, 1, Tq, Tk, 128, causal, seed=1400 + Tq)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_long_sequence(attn, d):
    # 9 key / query blocks per CTA walk: both stages of each kernel are reused many times
    _case(attn, 1, 4, 1, 1100, 1100, d, True, seed=1500 + d)


def test_backward_zero_upstream_gradient_and_determinism(attn):
    q, k, v = [t.to(DEV) for t in W.attention_inputs_custom(1, 4, 2, 300, 300, 128, 1600)]
    o, lse = attn.fwd(q, k, v, causal=True)
    z = attn.bwd(q, k, v, o, lse, torch.zeros_like(q), causal=True)
    torch.cuda.synchronize()
    assert all(torch.all(t == 0) for t in z)
    do = W.grad_output(1, 4, 300, 128, 1600).to(DEV)
    a = attn.bwd(q, k, v, o, lse, do, causal=True)
    b = attn.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_backward_outputs_offset_by_16_bytes(attn, d, causal):
    # 32-byte-aligned gradients are written with 32-byte stores (lane pairs swapping halves);
    # one gradient offset by 16 bytes sends all three through 16-byte stores: bitwise the same
    q, k, v = W.attention_inputs_custom(1, 4, 2, 333, 333, d, 4200 + d)
    do = W.grad_output(1, 4, 333, d, 4200 + d)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = attn.fwd(qd, kd, vd, causal=causal)
    ref = attn.bwd(qd, kd, vd, o, lse, dod, causal=causal)
    flat = torch.empty(k.numel() + 8, dtype=torch.bfloat16, device=DEV)
    dk16 = flat[8:].view(k.shape)
    assert dk16.data_ptr() % 32 == 16
    got = attn.bwd(qd, kd, vd, o, lse, dod, causal=causal, dk=dk16)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
