"""Parity of the CTA-pair prefill kernel (csrc/prefill_pair.cu, selected with
GB300_ATTN_PREFILL=pair) with the float64 oracle: every way the kernel groups four query
tiles into a unit (four heads of a K/V group at the same rows, two heads at two row tiles,
one head at four row tiles), both head sizes, causal and full masks, ragged tails and
rectangular Tq != Tk, and a sampled check at the full causal GQA B2 Hq32 Hkv8 T8192 d128
size. Tolerances as every other attention test (max |dO| <= 2e-2, mean |dO| <= 2e-3,
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
def pair_kernel(monkeypatch):
    monkeypatch.setenv("GB300_ATTN_PREFILL", "pair")


CASES = [  # B, Hq, Hkv, Tq, Tk, d, causal
    (1, 8, 2, 1000, 1000, 128, True),   # g = 4: four heads at the same rows
    (2, 4, 1, 333, 333, 128, False),
    (1, 8, 4, 700, 700, 128, True),     # g = 2: two heads at two row tiles (odd tile count)
    (1, 4, 2, 129, 129, 64, True),
    (2, 3, 3, 640, 640, 64, False),     # g = 1: one head at four row tiles
    (1, 2, 2, 900, 900, 64, True),
    (1, 2, 2, 100, 300, 128, True),     # rectangular, top-left causal
    (1, 4, 1, 300, 100, 64, False),
    (2, 8, 1, 1, 1, 128, True),         # a single key
    (1, 8, 2, 2200, 2200, 64, True),    # more key blocks than the d = 64 barrier ring (16)
    (1, 4, 1, 1300, 1300, 128, True),   # more key blocks than the d = 128 barrier ring (8)
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,causal", CASES)
def test_pair_kernel_matches_oracle(attn, pair_kernel, B, Hq, Hkv, Tq, Tk, d, causal):
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed=7 * Tq + d + Hq)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.attention(W.to_f64(q), W.to_f64(k), W.to_f64(v), causal, 1 / np.sqrt(d))
    assert_attn_close(o, lse, O, L, f"pair kernel B{B} Hq{Hq} Hkv{Hkv} Tq{Tq} Tk{Tk} d{d} causal={causal}")


def test_pair_kernel_equals_single_kernel_bitwise_at_small_size(attn, monkeypatch):
    # both kernels form S, P, l and O in the same order per row: identical bits
    q, k, v = [t.to(DEV) for t in W.attention_inputs_custom(1, 8, 2, 512, 512, 128, seed=5)]
    monkeypatch.setenv("GB300_ATTN_PREFILL", "single")
    o1, l1 = attn.fwd(q, k, v, causal=True)
    monkeypatch.setenv("GB300_ATTN_PREFILL", "pair")
    o2, l2 = attn.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_pair_kernel_full_size_sampled(attn, pair_kernel):
    shp = W.GQA_LLAMA
    q, k, v = W.attention_inputs(shp)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=shp.scale)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    rng = np.random.default_rng(31)
    g = shp.Hq // shp.Hkv
    for b, h in ((0, 0), (1, 31), (0, 13)):
        rows = np.sort(rng.choice(shp.T, 24, replace=False))
        rows[-1] = shp.T - 1
        O, L = oracle.attention_rows(W.to_f64(q[b:b + 1, h:h + 1]), W.to_f64(k[b:b + 1, h // g:h // g + 1]),
                                     W.to_f64(v[b:b + 1, h // g:h // g + 1]), 0, 0, rows, True, shp.scale)
        assert_attn_close(o[b, h, rows], lse[b, h, rows], O, L, f"pair kernel full size b{b} h{h}")
