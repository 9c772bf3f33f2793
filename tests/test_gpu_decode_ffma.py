"""Parity of the FFMA split kernel of flash-decoding (decode_split_kernel, selected with
GB300_ATTN_DECODE=ffma; the default split kernel runs on warp-level tensor-core MMAs) with
the float64 oracle: bf16 and E4M3 caches, both head sizes, the groupings of query heads per
CTA, lengths that end inside a stage, and equality (up to rounding) with the default kernel.
Tolerances as every other attention test (max |dO| <= 2e-2, mean |dO| <= 2e-3,
max |dLSE| <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import assert_attn_close, f64, require_gpu

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


@pytest.fixture
def ffma(monkeypatch):
    monkeypatch.setenv("GB300_ATTN_DECODE", "ffma")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (6, 2), (16, 2)])
def test_ffma_decode_matches_oracle(attn, ffma, d, Hq, Hkv):
    lens = [1, 17, 300, 1000]
    shp = W.DecodeShape("t", 4, Hq, Hkv, d, 1, 1000, 610 + Hq + d)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=lens)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=5)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), lens, shp.scale)
    assert_attn_close(o, lse, O, L, f"ffma decode d{d} Hq{Hq} Hkv{Hkv}")


@pytest.mark.parametrize("d", [64, 128])
def test_ffma_decode_fp8_matches_oracle(attn, ffma, d):
    lens = [5, 64, 700]
    shp = W.DecodeShape("t", 3, 8, 2, d, 1, 700, 620 + d)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=lens)
    kq, ks = attn.kv_quantize_fp8(kc.to(DEV))
    vq, vs = attn.kv_quantize_fp8(vc.to(DEV))
    o, lse = attn.decode_fp8(q.to(DEV), kq, vq, ks, vs, sl.to(DEV), num_splits=3)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    # the oracle quantises the bf16 cache itself (the GPU's codes are byte-exact with its own,
    # tested in test_gpu_parity.py) and decodes its codes
    okc, oks = oracle.quantize_kv(f64(kc))
    ovc, ovs = oracle.quantize_kv(f64(vc))
    O, L = oracle.decode_fp8(f64(q), okc, ovc, oks, ovs, lens, shp.scale)
    assert_attn_close(o, lse, O, L, f"ffma E4M3 decode d{d}")


def test_ffma_and_mma_decode_agree(attn, monkeypatch):
    shp = W.DecodeShape("t", 8, 32, 8, 128, 100, 3000, 630)
    q, kc, vc, sl = [t.to(DEV) for t in W.decode_inputs(shp)]
    monkeypatch.setenv("GB300_ATTN_DECODE", "ffma")
    o1, l1 = attn.decode(q, kc, vc, sl, num_splits=4)
    monkeypatch.setenv("GB300_ATTN_DECODE", "mma")
    o2, l2 = attn.decode(q, kc, vc, sl, num_splits=4)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3
