"""Parity at the full workload sizes, in the launch configuration bench.py times,
on sampled outputs that the float64 oracle computes row by row; plus long
sequences that wrap the prefill kernel's K/V slot ring and barrier rings many
times for both head dims.

Sampled rows always include the first and last row, rows on both sides of
128-row tile boundaries, and random rows, for a spread of (batch, head) pairs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import assert_attn_close, assert_norm_close, f64, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


def _sample_rows(T, seed, n_random=24):
    rng = np.random.default_rng(seed)
    rows = {0, 1, T - 1, T - 2}
    for t in (127, 128, 129, T // 2 - 1, T // 2, T - 129, T - 128):
        if 0 <= t < T:
            rows.add(t)
    rows.update(rng.integers(0, T, size=n_random).tolist())
    return np.array(sorted(rows))


def _check_sampled(q, k, v, o, lse, causal, scale, pairs, seed):
    O_all, L_all, o_all, l_all = [], [], [], []
    for i, (b, h) in enumerate(pairs):
        rows = _sample_rows(q.shape[2], seed + i)
        qh = f64(q[b:b + 1, h:h + 1])
        g = q.shape[1] // k.shape[1]
        kh = f64(k[b:b + 1, h // g:h // g + 1])
        vh = f64(v[b:b + 1, h // g:h // g + 1])
        Or, Lr = oracle.attention_rows(qh, kh, vh, 0, 0, rows, causal, scale)
        O_all.append(Or)
        L_all.append(Lr)
        o_all.append(f64(o[b, h, rows]))
        l_all.append(f64(lse[b, h, rows]))
    return assert_attn_close(np.concatenate(o_all), np.concatenate(l_all), np.concatenate(O_all),
                             np.concatenate(L_all), "sampled rows")


@pytest.mark.parametrize("shape", [W.MHA_GPT2, W.GQA_QWEN, W.GQA_LLAMA], ids=["mha-gpt2", "gqa-qwen", "gqa-llama"])
def test_prefill_full_size_sampled(attn, shape):
    q, k, v = W.attention_inputs(shape)[:3]
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=shape.causal, scale=shape.scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(shape.seed)
    pairs = {(0, 0), (shape.B - 1, shape.Hq - 1), (0, shape.Hq // 2)}
    for _ in range(5):
        pairs.add((int(rng.integers(shape.B)), int(rng.integers(shape.Hq))))
    _check_sampled(q, k, v, o, lse, shape.causal, shape.scale, sorted(pairs), shape.seed)


@pytest.mark.parametrize("shape,group", [(W.GQA_LLAMA, (1, 5)), (W.GQA_QWEN, (0, 3))], ids=["gqa-llama", "gqa-qwen"])
def test_backward_full_size_sampled(attn, shape, group):
    # the full backward on the workload; the oracle checks sampled dQ rows of every query head of
    # one K/V group and sampled dK, dV rows of that K/V head (tolerance as tests/test_gpu_backward.py)
    q, k, v = W.attention_inputs(shape)[:3]
    do = W.grad_output(shape.B, shape.Hq, shape.T, shape.d, shape.seed)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = attn.fwd(qd, kd, vd, causal=shape.causal, scale=shape.scale)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, lse, dod, causal=shape.causal, scale=shape.scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    b, kvh = group
    g = shape.Hq // shape.Hkv
    rows = _sample_rows(shape.T, shape.seed + 77, n_random=12)
    sl = slice(b, b + 1)
    rq, rk, rv = oracle.attention_backward_rows(f64(q[sl]), f64(k[sl]), f64(v[sl]), f64(do[sl]), shape.causal,
                                                shape.scale, 0, kvh, rows, rows)
    got_q = f64(dq[b, kvh * g:(kvh + 1) * g][:, rows])
    for name, got, want in (("dQ", got_q, rq), ("dK", f64(dk[b, kvh, rows]), rk), ("dV", f64(dv[b, kvh, rows]), rv)):
        err = np.abs(got - want)
        assert np.all(np.isfinite(got)), name
        assert err.max() <= 2e-2 * np.abs(want).max() + 1e-6, (name, err.max(), np.abs(want).max())
        assert err.mean() <= 1e-2 * np.abs(want).mean() + 1e-7, (name, err.mean(), np.abs(want).mean())


def test_decode_full_size(attn):
    shp = W.DECODE_LLAMA
    q, kc, vc, sl = W.decode_inputs(shp)
    S = attn.default_splits(shp.B, shp.Hkv, shp.Lcap)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=S)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = f64(o), f64(lse)
    O = np.empty_like(o)
    L = np.empty_like(lse)
    for b in range(shp.B):  # one sequence at a time keeps the float64 copies small
        Ob, Lb = oracle.decode(f64(q[b:b + 1]), f64(kc[b:b + 1]), f64(vc[b:b + 1]), sl[b:b + 1].numpy(), shp.scale)
        O[b], L[b] = Ob[0], Lb[0]
    assert_attn_close(o, lse, O, L, "decode full size")


def test_decode_fp8_full_size(attn):
    # the decode workload with its cache quantised to E4M3 on the GPU; the oracle quantises the
    # sampled sequences itself (all their heads) and decodes them
    shp = W.DECODE_LLAMA
    q, kc, vc, sl = W.decode_inputs(shp)
    kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
    vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
    S = attn.default_splits(shp.B, shp.Hkv, shp.Lcap)
    o, lse = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=S)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = f64(o), f64(lse)
    for b in (0, shp.B - 1):
        okc, oks = oracle.quantize_kv(f64(kc[b:b + 1]))
        ovc, ovs = oracle.quantize_kv(f64(vc[b:b + 1]))
        assert np.array_equal(ksc[b].cpu().numpy(), oks[0]) and np.array_equal(vsc[b].cpu().numpy(), ovs[0])
        assert np.array_equal(kcodes[b, 0].cpu().numpy(), okc[0, 0])
        Ob, Lb = oracle.decode_fp8(f64(q[b:b + 1]), okc, ovc, oks, ovs, sl[b:b + 1].numpy(), shp.scale)
        assert_attn_close(o[b:b + 1], lse[b:b + 1], Ob, Lb, f"fp8 decode full size, sequence {b}")


def test_rmsnorm_full_size(attn):
    x, w = W.norm_inputs(W.NORM_QWEN)
    y = attn.rmsnorm(x.to(DEV), w.to(DEV), eps=W.NORM_QWEN.eps)
    torch.cuda.synchronize()
    assert_norm_close(y, oracle.rmsnorm(f64(x), f64(w), W.NORM_QWEN.eps), "X[4096,1024]")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,T", [(2, 1, 2100), (4, 2, 1536), (3, 3, 1100)])
def test_prefill_long_sequences_wrap_the_rings(attn, d, causal, Hq, Hkv, T):
    # 9 to 17 key blocks per query tile: more than the 11-slot (d=64) / 5-slot (d=128)
    # K/V ring and the 8-deep per-block barrier rings
    q, k, v = W.attention_inputs_custom(1, Hq, Hkv, T, T, d, seed=600 + T + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), causal, scale)
    assert_attn_close(o, lse, O, L, f"T{T} d{d} Hq{Hq} Hkv{Hkv} causal{causal}")


def test_prefill_long_context_sampled(attn):
    # one sequence of 65 536 tokens (causal GQA, d = 128): rows near the end accumulate 512 key blocks
    B, Hq, Hkv, T, d = 1, 4, 1, 65536, 128
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, T, T, d, 4242)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check_sampled(q, k, v, o, lse, True, scale, [(0, 0), (0, 3)], 4242)


def test_decode_long_context(attn):
    # caches of 131 072 tokens, one sequence full and one not
    shp = W.DecodeShape("long", 2, 8, 2, 128, 1, 131072, 4343)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=[131072, 100001])
    S = attn.default_splits(shp.B, shp.Hkv, shp.Lcap)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=S)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), shp.scale)
    assert_attn_close(o, lse, O, L, f"decode long context, {S} splits")
