"""Pins of the oracle's backward pass against things other than itself: PyTorch
autograd in float64 through an ordinary masked-softmax attention (an independent
differentiation of the forward, the check the source page itself runs:
"FlashAttention: attention without the n x n matrix", section "Backward pass:
recomputing is cheaper than storing"), central finite differences of the oracle's
own forward on a tiny case, and closed forms (constant values, one key, zero
upstream gradient)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _inputs(B, Hq, Hkv, Tq, Tk, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Tq, d))
    k = rng.standard_normal((B, Hkv, Tk, d))
    v = rng.standard_normal((B, Hkv, Tk, d))
    do = rng.standard_normal((B, Hq, Tq, d))
    return q, k, v, do


def _oracle_grads(q, k, v, do, causal, scale):
    o, lse = oracle.attention(q, k, v, causal, scale)
    return oracle.attention_backward(q, k, v, o, lse, do, causal, scale)


def _autograd_grads(q, k, v, do, causal, scale):
    Q, K, V = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    g = q.shape[1] // k.shape[1]
    Kx, Vx = K.repeat_interleave(g, dim=1), V.repeat_interleave(g, dim=1)
    S = Q @ Kx.transpose(-1, -2) * scale
    if causal:
        Tq, Tk = q.shape[2], k.shape[2]
        mask = torch.ones(Tq, Tk, dtype=torch.bool).tril()
        S = S.masked_fill(~mask, float("-inf"))
    O = torch.softmax(S, dim=-1) @ Vx
    O.backward(torch.tensor(do))
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,causal", [
    (1, 1, 1, 64, 64, 16, True),     # the page's own check: T = 64, d = 16, causal
    (2, 4, 2, 37, 37, 8, True),      # GQA g = 2, ragged length
    (1, 3, 1, 20, 33, 8, False),     # g = 3, rectangular, no mask
    (1, 2, 2, 33, 20, 8, True),      # Tq > Tk, top-left causal
])
def test_backward_matches_float64_autograd(B, Hq, Hkv, Tq, Tk, d, causal):
    q, k, v, do = _inputs(B, Hq, Hkv, Tq, Tk, d, seed=B * 100 + Tq + d)
    scale = 1.0 / math.sqrt(d)
    mine = _oracle_grads(q, k, v, do, causal, scale)
    ref = _autograd_grads(q, k, v, do, causal, scale)
    for name, a, b in zip(("dQ", "dK", "dV"), mine, ref):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max()), name


def test_backward_matches_finite_differences():
    q, k, v, do = _inputs(1, 2, 1, 5, 5, 3, seed=9)
    scale, eps = 0.7, 1e-6
    dq, dk, dv = _oracle_grads(q, k, v, do, True, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.attention(qq, kk, vv, True, scale)
        return float(np.sum(o * do))

    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            up = loss(q, k, v)
            arr[idx] = old - eps
            dn = loss(q, k, v)
            arr[idx] = old
            assert abs((up - dn) / (2 * eps) - grad[idx]) <= 1e-7


def test_backward_closed_forms():
    q, k, v, do = _inputs(1, 2, 1, 6, 6, 4, seed=11)
    scale = 0.5
    # zero upstream gradient: every gradient is zero
    z = _oracle_grads(q, k, v, np.zeros_like(do), True, scale)
    assert all(np.array_equal(t, np.zeros_like(t)) for t in z)
    # equal value rows: O_i = c for every row, dS = P (dO_i.c - dO_i.c) = 0, so dQ = dK = 0 and
    # dV_j = sum over the query heads and rows of P_ij dO_i
    vc = np.repeat(v[:, :, :1], 6, axis=2)
    dq, dk, dv = _oracle_grads(q, k, vc, do, True, scale)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    o, lse = oracle.attention(q, k, vc, True, scale)
    s = np.einsum("bhid,bjd->bhij", q, k[:, 0]) * scale
    s = np.where(np.tril(np.ones((6, 6), dtype=bool)), s, -np.inf)
    p = np.exp(s - lse[..., None])
    assert np.allclose(dv[0, 0], np.einsum("hij,hid->jd", p[0], do[0]), atol=1e-12)
    # a single key (no mask): P = 1, dV_0 = sum of dO over heads and rows, dQ = dK = 0
    q1, k1, v1, do1 = _inputs(1, 2, 1, 4, 1, 4, seed=12)
    dq, dk, dv = _oracle_grads(q1, k1, v1, do1, False, scale)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.allclose(dv[0, 0, 0], do1[0].sum(axis=(0, 1)), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_match_the_full_gradients(causal):
    # the sampled-row form used at full sizes against the pinned full gradients
    q, k, v, do = _inputs(2, 6, 2, 50, 50, 8, seed=13)
    scale = 0.4
    dq, dk, dv = _oracle_grads(q, k, v, do, causal, scale)
    qr, kr = [0, 7, 31, 49], [0, 1, 25, 49]
    for b, kvh in ((0, 0), (1, 1)):
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, causal, scale, b, kvh, qr, kr)
        for gi in range(3):
            assert np.allclose(rq[gi], dq[b, kvh * 3 + gi, qr], atol=1e-12)
        assert np.allclose(rk, dk[b, kvh, kr], atol=1e-12) and np.allclose(rv, dv[b, kvh, kr], atol=1e-12)
