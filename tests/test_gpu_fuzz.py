"""Randomised parity sweep: seeded random shapes for prefill, backward and decode against the
float64 oracle, at the tolerances of the other parity tests.

The fixed tests pick shapes by hand (tile edges, tails, groupings). Here the shapes are drawn
from a fixed seed, so that the combinations nobody picked get covered too:
* batch and head counts, with the query heads a multiple of the K/V heads;
* Tq != Tk on both sides of each other, including lengths below, at and past a tile;
* causal and not, d = 64 and 128; the output 32-byte aligned or offset by 16 bytes;
* decode lengths anywhere in [1, Lcap] and split counts up to Lcap / 16, for the bf16 and the
  E4M3 cache, and the balanced schedule (num_splits = 0) over lengths from 0 to Lcap;
* non-causal prefill with the persistent CTA count capped at random, so that the last round's
  units are split along the keys and merged;
* RMSNorm rows and widths on both sides of the block-per-row threshold, with and without the
  residual add.

The draws are reproducible; a failure names its case.
"""
import math
import random

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import assert_attn_close, assert_norm_close, bf16_round, f64, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


def _attn_cases(n, seed, max_t):
    rnd = random.Random(seed)
    for _ in range(n):
        Hkv = rnd.choice([1, 1, 2, 3])
        g = rnd.choice([1, 2, 3, 4])
        B = rnd.choice([1, 1, 2, 3])
        Tq = rnd.choice([rnd.randint(1, 130), rnd.randint(1, max_t)])
        Tk = rnd.choice([Tq, rnd.randint(1, max_t)])
        d = rnd.choice([64, 128])
        causal = rnd.choice([False, True])
        yield B, Hkv * g, Hkv, Tq, Tk, d, causal, rnd.randint(0, 10**6)


@pytest.mark.parametrize("case", list(_attn_cases(48, 2024, 700)), ids=lambda c: "B{}_Hq{}_Hkv{}_Tq{}_Tk{}_d{}_c{}".format(*c[:7]))
def test_prefill_random_shapes(attn, case):
    B, Hq, Hkv, Tq, Tk, d, causal, seed = case
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed)
    scale = 1.0 / math.sqrt(d)
    # O either 32-byte aligned (32-byte stores) or offset by 16 bytes (16-byte stores)
    off = 8 if seed % 2 else 0
    flat = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=DEV)
    out = flat[off:off + q.numel()].view(q.shape)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, out=out)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), causal, scale)
    assert_attn_close(o, lse, O, L, f"prefill {case[:7]} O offset {2 * off} B")


def _grad_close(got, want, what):
    got = f64(got)
    err = np.abs(got - want)
    scale_max, scale_mean = np.abs(want).max(), np.abs(want).mean()
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max() <= 2e-2 * scale_max + 1e-6, f"{what}: max err {err.max():.3e} vs max |ref| {scale_max:.3e}"
    assert err.mean() <= 1e-2 * scale_mean + 1e-7, f"{what}: mean err {err.mean():.3e} vs mean |ref| {scale_mean:.3e}"


@pytest.mark.parametrize("case", list(_attn_cases(32, 4048, 400)), ids=lambda c: "B{}_Hq{}_Hkv{}_Tq{}_Tk{}_d{}_c{}".format(*c[:7]))
def test_backward_random_shapes(attn, case):
    B, Hq, Hkv, Tq, Tk, d, causal, seed = case
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed)
    do = W.grad_output(B, Hq, Tq, d, seed)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = attn.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, lse, do.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    qf, kf, vf = f64(q), f64(k), f64(v)
    O, L = oracle.attention(qf, kf, vf, causal, scale)
    dQ, dK, dV = oracle.attention_backward(qf, kf, vf, O, L, f64(do), causal, scale)
    tag = f"backward {case[:7]}"
    _grad_close(dq, dQ, "dQ " + tag)
    _grad_close(dk, dK, "dK " + tag)
    _grad_close(dv, dV, "dV " + tag)


def _decode_cases(n, seed):
    rnd = random.Random(seed)
    for _ in range(n):
        Hkv = rnd.choice([1, 2, 4, 8])
        g = rnd.choice([1, 2, 3, 4, 6])
        B = rnd.randint(1, 6)
        Lcap = rnd.choice([rnd.randint(1, 64), rnd.randint(16, 3000)])
        lens = [rnd.randint(1, Lcap) for _ in range(B)]
        d = rnd.choice([64, 128])
        smax = max(1, (Lcap + 15) // 16)
        S = rnd.randint(1, min(smax, 64))
        yield B, Hkv * g, Hkv, d, Lcap, tuple(lens), S, rnd.randint(0, 10**6)


@pytest.mark.parametrize("case", list(_decode_cases(48, 8096)), ids=lambda c: "B{}_Hq{}_Hkv{}_d{}_L{}_S{}".format(c[0], c[1], c[2], c[3], c[4], c[6]))
def test_decode_random_shapes(attn, case):
    B, Hq, Hkv, d, Lcap, lens, S, seed = case
    shp = W.DecodeShape("fuzz", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=list(lens))
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=S)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), shp.scale)
    assert_attn_close(o, lse, O, L, f"decode {case[:7]}")


@pytest.mark.parametrize("case", list(_decode_cases(24, 16192)), ids=lambda c: "B{}_Hq{}_Hkv{}_d{}_L{}_S{}".format(c[0], c[1], c[2], c[3], c[4], c[6]))
def test_decode_fp8_random_shapes(attn, case):
    # the cache quantised on the GPU (codes byte-exact with the oracle's, tested elsewhere), then
    # decoded; the oracle decodes its own codes and scales
    B, Hq, Hkv, d, Lcap, lens, S, seed = case
    shp = W.DecodeShape("fuzz", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=list(lens))
    kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
    vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
    o, lse = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=S)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    okc, oks = oracle.quantize_kv(f64(kc))
    ovc, ovs = oracle.quantize_kv(f64(vc))
    O, L = oracle.decode_fp8(f64(q), okc, ovc, oks, ovs, sl.numpy(), shp.scale)
    assert_attn_close(o, lse, O, L, f"fp8 decode {case[:7]}")


def _balanced_cases(n, seed):
    rnd = random.Random(seed)
    for _ in range(n):
        Hkv = rnd.choice([1, 2, 4, 8])
        g = rnd.choice([1, 2, 3, 4, 6, 8])
        B = rnd.randint(1, 12)
        Lcap = rnd.choice([rnd.randint(1, 200), rnd.randint(16, 5000)])
        lens = [rnd.choice([0, 1, rnd.randint(1, Lcap), Lcap]) for _ in range(B)]
        yield B, Hkv * g, Hkv, rnd.choice([64, 128]), Lcap, tuple(lens), rnd.random() < 0.5, rnd.randint(0, 10**6)


@pytest.mark.parametrize("case", list(_balanced_cases(40, 24601)),
                         ids=lambda c: "B{}_Hq{}_Hkv{}_d{}_L{}_fp8{}".format(c[0], c[1], c[2], c[3], c[4], int(c[6])))
def test_decode_balanced_random_shapes(attn, case):
    B, Hq, Hkv, d, Lcap, lens, fp8, seed = case
    shp = W.DecodeShape("fuzz", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=[max(1, x) for x in lens])
    sl = torch.tensor(lens, dtype=torch.int32)  # zero lengths too: O = 0, LSE = -inf
    if fp8:
        kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
        vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
        o, lse = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=0)
    else:
        o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = f64(o), f64(lse)
    zero = [b for b in range(B) if lens[b] == 0]
    for b in zero:
        assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b])), f"empty sequence {b}"
    keep = [b for b in range(B) if lens[b] > 0]
    if not keep:
        return
    if fp8:
        okc, oks = oracle.quantize_kv(f64(kc))
        ovc, ovs = oracle.quantize_kv(f64(vc))
        O, L = oracle.decode_fp8(f64(q)[keep], okc[keep], ovc[keep], oks[keep], ovs[keep], sl.numpy()[keep], shp.scale)
    else:
        O, L = oracle.decode(f64(q)[keep], f64(kc)[keep], f64(vc)[keep], sl.numpy()[keep], shp.scale)
    assert_attn_close(o[keep], lse[keep], O, L, f"balanced decode {case[:7]}")


def _split_prefill_cases(n, seed):
    rnd = random.Random(seed)
    for _ in range(n):
        Hkv = rnd.choice([1, 2, 3])
        g = rnd.choice([1, 2, 3, 4])
        B = rnd.choice([1, 2, 3])
        Tq = rnd.randint(1, 1200)
        Tk = rnd.choice([Tq, rnd.randint(1, 2500)])
        yield B, Hkv * g, Hkv, Tq, Tk, rnd.choice([64, 128]), rnd.randint(1, 24), rnd.randint(0, 10**6)


@pytest.mark.parametrize("case", list(_split_prefill_cases(32, 51200)),
                         ids=lambda c: "B{}_Hq{}_Hkv{}_Tq{}_Tk{}_d{}_ctas{}".format(*c[:7]))
def test_prefill_split_tail_random_shapes(attn, monkeypatch, case):
    B, Hq, Hkv, Tq, Tk, d, ctas, seed = case
    monkeypatch.setenv("GB300_ATTN_PREFILL_CTAS", str(ctas))
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=False, scale=scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), False, scale)
    assert_attn_close(o, lse, O, L, f"split-tail prefill {case[:7]}")


def _norm_cases(n, seed):
    rnd = random.Random(seed)
    for _ in range(n):
        if rnd.random() < 0.5:
            D = 64 * rnd.randint(1, 128)             # 8 segments, up to 8192
        else:
            D = 8 * rnd.randint(1, 512)              # any multiple of 8 up to 4096
        T = rnd.choice([rnd.randint(1, 8), rnd.randint(1, 600), rnd.randint(500, 3000)])
        yield T, D, rnd.random() < 0.5, rnd.randint(0, 10**6)


@pytest.mark.parametrize("case", list(_norm_cases(32, 32384)), ids=lambda c: "T{}_D{}_res{}".format(*c[:3]))
def test_rmsnorm_random_shapes(attn, case):
    T, D, residual, seed = case
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, D, generator=gen).to(torch.bfloat16)
    w = (0.5 + torch.rand(D, generator=gen)).to(torch.bfloat16)
    if residual:
        r = torch.randn(T, D, generator=gen).to(torch.bfloat16)
        y, h = attn.rmsnorm_residual(x.to(DEV), r.to(DEV), w.to(DEV), eps=1e-6)
        torch.cuda.synchronize()
        # h is the exact sum rounded once to bf16; y normalises that stored h
        assert np.array_equal(f64(h), bf16_round(f64(x) + f64(r))), f"h T{T} D{D}"
        assert_norm_close(y, oracle.rmsnorm(f64(h), f64(w), 1e-6), f"residual T{T} D{D}")
    else:
        y = attn.rmsnorm(x.to(DEV), w.to(DEV), eps=1e-6)
        torch.cuda.synchronize()
        assert_norm_close(y, oracle.rmsnorm(f64(x), f64(w), 1e-6), f"T{T} D{D}")
