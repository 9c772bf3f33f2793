"""Seeded synthetic inputs for the attention / decode / RMSNorm workloads.

This module only draws random numbers and fixes shapes. It holds none of the
method's arithmetic, so both the float64 oracle (``oracle/``) and the CUDA
path (``exact_tiled_attention_attn_gb300``) can be fed from it without sharing
any computation.

Recipe (all tensors are drawn on the CPU with one ``torch.Generator`` per
workload, in the order listed, as float32 N(0, 1) and then rounded once to
bfloat16 with round-to-nearest-even):

* attention: q [B, Hq, T, d], k [B, Hkv, T, d], v [B, Hkv, T, d]
* RMSNorm:   x [T, D] ~ N(0, 1);  w [D] ~ U(0.5, 1.5)
* decode:    q [B, Hq, d], kcache / vcache [B, Hkv, Lcap, d], and per-sequence
  lengths drawn with ``numpy.random.default_rng(seed)`` uniformly in
  [Lmin, Lmax] (both ends included).

The shapes are the head layouts the pages use as examples (GPT-2-small-like
12 heads x 64, Qwen3-0.6B-like 16/8 heads x 128, Llama-3-8B-like 32/8 heads x
128); no weights or datasets are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class AttnShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    d: int
    causal: bool
    seed: int
    fp32_inputs: bool = False  # the single-head case is specified with fp32 inputs

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs that take part (causal: j <= i)."""
        per_head = self.T * (self.T + 1) // 2 if self.causal else self.T * self.T
        return self.B * self.Hq * per_head

    def flops(self) -> float:
        """Algorithmic FLOPs: 2d for q.k plus 2d for p.v per visible pair."""
        return 4.0 * self.d * self.visible_pairs()

    def hbm_bytes(self) -> int:
        """Compulsory HBM bytes: read Q, K, V once, write O (bf16) and LSE (fp32)."""
        q = self.B * self.Hq * self.T * self.d * 2
        kv = 2 * self.B * self.Hkv * self.T * self.d * 2
        lse = self.B * self.Hq * self.T * 4
        return 2 * q + kv + lse


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    Lmin: int
    Lmax: int
    seed: int

    @property
    def Lcap(self) -> int:
        return self.Lmax

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class NormShape:
    name: str
    T: int
    D: int
    eps: float
    seed: int

    def hbm_bytes(self) -> int:
        return 2 * self.T * self.D * 2 + self.D * 2


# The five workloads of the specification, in order.
SINGLE_HEAD = AttnShape("single-head causal B1 H1 T256 d64 (fp32 inputs rounded to bf16)",
                        1, 1, 1, 256, 64, True, 1000, fp32_inputs=True)
MHA_GPT2 = AttnShape("non-causal MHA B8 H12 T4096 d64", 8, 12, 12, 4096, 64, False, 1001)
GQA_QWEN = AttnShape("causal GQA B1 Hq16 Hkv8 T4096 d128", 1, 16, 8, 4096, 128, True, 1002)
NORM_QWEN = NormShape("RMSNorm X[4096,1024] eps 1e-6", 4096, 1024, 1e-6, 1002)
GQA_LLAMA = AttnShape("causal GQA B2 Hq32 Hkv8 T8192 d128", 2, 32, 8, 8192, 128, True, 1003)
DECODE_LLAMA = DecodeShape("flash-decoding B16 Hq32 Hkv8 d128 L~U[8192,32768]",
                           16, 32, 8, 128, 8192, 32768, 1004)

ATTN_WORKLOADS = (SINGLE_HEAD, MHA_GPT2, GQA_QWEN, GQA_LLAMA)


def _randn(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def attention_inputs(shape: AttnShape, T: int | None = None, q_scale: float = 1.0,
                     seed: int | None = None):
    """Return (q, k, v) bf16 CPU tensors in [B, H, T, d] layout.

    ``T`` overrides the sequence length (small parity cases), ``q_scale``
    multiplies q before rounding (the peaked-softmax stability case).
    For the fp32-specified workload the fp32 draws are returned too, as a
    fourth element, for an information-only comparison.
    """
    T = shape.T if T is None else T
    gen = torch.Generator().manual_seed(shape.seed if seed is None else seed)
    q32 = _randn(gen, (shape.B, shape.Hq, T, shape.d)) * q_scale
    k32 = _randn(gen, (shape.B, shape.Hkv, T, shape.d))
    v32 = _randn(gen, (shape.B, shape.Hkv, T, shape.d))
    out = (q32.to(torch.bfloat16), k32.to(torch.bfloat16), v32.to(torch.bfloat16))
    if shape.fp32_inputs:
        return out + ((q32, k32, v32),)
    return out


def attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed, q_scale: float = 1.0):
    """Free-shape variant used by edge-case tests (Tq may differ from Tk)."""
    gen = torch.Generator().manual_seed(seed)
    q = (_randn(gen, (B, Hq, Tq, d)) * q_scale).to(torch.bfloat16)
    k = _randn(gen, (B, Hkv, Tk, d)).to(torch.bfloat16)
    v = _randn(gen, (B, Hkv, Tk, d)).to(torch.bfloat16)
    return q, k, v


def grad_output(B, Hq, Tq, d, seed):
    """The upstream gradient dO [B, Hq, Tq, d] for the backward pass: N(0,1) rounded to bf16,
    from its own generator (seed + 7919, so it differs from the forward inputs' draws)."""
    gen = torch.Generator().manual_seed(seed + 7919)
    return _randn(gen, (B, Hq, Tq, d)).to(torch.bfloat16)


def norm_inputs(shape: NormShape, T: int | None = None, seed: int | None = None):
    T = shape.T if T is None else T
    gen = torch.Generator().manual_seed(shape.seed if seed is None else seed)
    x = _randn(gen, (T, shape.D)).to(torch.bfloat16)
    w = (0.5 + torch.rand(shape.D, generator=gen, dtype=torch.float32)).to(torch.bfloat16)
    return x, w


def decode_lengths(shape: DecodeShape, B: int | None = None, seed: int | None = None) -> np.ndarray:
    B = shape.B if B is None else B
    rng = np.random.default_rng(shape.seed if seed is None else seed)
    return rng.integers(shape.Lmin, shape.Lmax, size=B, endpoint=True).astype(np.int32)


def decode_inputs(shape: DecodeShape, B: int | None = None, Lcap: int | None = None,
                  seqlens=None, seed: int | None = None):
    """Return (q [B,Hq,d], kcache [B,Hkv,Lcap,d], vcache, seqlens int32 [B]).

    The whole cache (Lcap rows per sequence) is filled with N(0,1) draws;
    only the first ``seqlens[b]`` rows of sequence b take part.
    """
    B = shape.B if B is None else B
    Lcap = shape.Lcap if Lcap is None else Lcap
    if seqlens is None:
        seqlens = decode_lengths(shape, B, seed)
    seqlens = np.asarray(seqlens, dtype=np.int32)
    gen = torch.Generator().manual_seed(shape.seed if seed is None else seed)
    q = _randn(gen, (B, shape.Hq, shape.d)).to(torch.bfloat16)
    kc = torch.empty((B, shape.Hkv, Lcap, shape.d), dtype=torch.bfloat16)
    vc = torch.empty((B, shape.Hkv, Lcap, shape.d), dtype=torch.bfloat16)
    # Draw per sequence to keep the peak float32 temporary small.
    for b in range(B):
        kc[b] = _randn(gen, (shape.Hkv, Lcap, shape.d)).to(torch.bfloat16)
        vc[b] = _randn(gen, (shape.Hkv, Lcap, shape.d)).to(torch.bfloat16)
    return q, kc, vc, torch.from_numpy(seqlens.copy())


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Decode a (bf16 / fp32) CPU tensor exactly to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
