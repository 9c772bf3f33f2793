"""FP8 E4M3 codes, a KV cache quantised with one scale per (sequence, K/V head), and
flash-decoding over that cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definitions followed:

* The E4M3 format ("Chapter 5. Operators and runtime", section 5.4.3, example
  5-7; "How does FlashAttention-3 work mathematically", section 6, FP8 support:
  E4M3 for K and V): one sign bit, four exponent bits, three mantissa bits, the
  largest finite magnitude 448. Written out: exponent bias 7; an exponent field
  e > 0 encodes (1 + m/8) * 2^(e - 7), e = 0 encodes the subnormals
  (m/8) * 2^-6; there are no infinities, and the one code with every exponent
  and mantissa bit set (per sign) is NaN, which is what makes 448 = 1.75 * 2^8
  the largest finite value.
* Quantisation with a scale (the same example): the scale maps the largest
  magnitude of the block it covers onto 448; each element is divided by the
  scale, rounded to a representable value, and dequantised by multiplying the
  code's value by the scale again. Example 5-7 rounds 44.8 to 44, i.e. to the
  nearest representable value; ties go to the even mantissa (the usual IEEE
  rule), and magnitudes above 448 saturate to 448.
* Precision of the scale arithmetic (the pages leave it open; the plainest
  reading for a cache written by a GPU kernel): scale = amax / 448 and x / scale
  are each one correctly rounded float32 division; the rounding to E4M3 is
  exact on that float32 quotient. One scale per (sequence, K/V head) over its
  whole [L, d] block ("per-head scale"); an all-zero block gets scale 1.
* Decode over the quantised cache = the exact decode of ``oracle.decode`` on
  the dequantised keys and values ("Attention from the kernel's side", section
  "Why a quantised cache needs a fused kernel": the values are dequantised in
  registers while the tile is loaded, so the attention itself is unchanged).
"""
from __future__ import annotations

import numpy as np

from .attention import decode

E4M3_MAX = 448.0
_NAN_CODES = (0x7F, 0xFF)


def e4m3_value(code: int) -> float:
    """The real number an E4M3 code stands for (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    if code in _NAN_CODES:
        return float("nan")
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    """float64 [256]: the value of every code."""
    return np.array([e4m3_value(c) for c in range(256)])


_TABLE = e4m3_table()
# non-negative finite codes 0x00..0x7E in increasing order of value
_POS_CODES = np.arange(0x7F)
_POS_VALUES = _TABLE[:0x7F]


def e4m3_encode(x) -> np.ndarray:
    """Round each element to the nearest E4M3 value: ties to the even mantissa,
    magnitudes above 448 saturate to 448, NaN -> 0x7F, the sign of zero kept.

    Written as a search over the 127 non-negative finite values (sorted by code),
    so that it follows the definition rather than any bit trick.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    hi = np.searchsorted(_POS_VALUES, a)                 # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _POS_VALUES[lo]
    dhi = _POS_VALUES[hi] - a
    exact = dhi == 0
    pick_lo = (dlo < dhi) | ((dlo == dhi) & ((lo & 1) == 0))   # nearer, or a tie with an even mantissa
    code = np.where(exact, hi, np.where(pick_lo, lo, hi)).astype(np.uint8)
    code = code | np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def head_scale(block) -> np.float32:
    """The scale of one block: amax / 448 as one float32 division; 1 for an all-zero block."""
    amax = np.float32(np.max(np.abs(np.asarray(block, dtype=np.float64)))) if np.size(block) else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax) / np.float32(E4M3_MAX)


def quantize_block(block, scale: np.float32) -> np.ndarray:
    """E4M3 codes of block / scale, the quotient taken as one float32 division."""
    quot = np.asarray(block, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(quot.astype(np.float64))


def quantize_kv(x) -> tuple[np.ndarray, np.ndarray]:
    """x: [B, H, L, d] (float64 values of bf16 numbers). Returns codes uint8 [B, H, L, d]
    and scales float32 [B, H], one per (sequence, head) over its whole [L, d] block."""
    x = np.asarray(x, dtype=np.float64)
    B, H = x.shape[:2]
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((B, H), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            sc = head_scale(x[b, h])
            scales[b, h] = sc
            codes[b, h] = quantize_block(x[b, h], sc)
    return codes, scales


def dequantize_kv(codes, scales) -> np.ndarray:
    """float64 [B, H, L, d]: value(code) * scale (exact in float64)."""
    vals = _TABLE[np.asarray(codes, dtype=np.uint8)]
    return vals * np.asarray(scales, dtype=np.float64)[:, :, None, None]


def decode_fp8(q, kcodes, vcodes, kscales, vscales, seqlens, scale: float):
    """Single-query attention over an E4M3 KV cache: the exact decode on the
    dequantised keys and values. q [B, Hq, d]; codes [B, Hkv, Lcap, d]; scales
    [B, Hkv]. Returns O [B, Hq, d] and LSE [B, Hq]."""
    return decode(q, dequantize_kv(kcodes, kscales), dequantize_kv(vcodes, vscales), seqlens, scale)
