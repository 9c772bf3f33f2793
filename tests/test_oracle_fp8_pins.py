"""Pins of the FP8 (E4M3) part of the oracle against things other than itself:
the worked example printed in "Chapter 5. Operators and runtime" (section 5.4.3,
example 5-7), PyTorch's own float8_e4m3fn dtype as an independent library
implementation of the format, closed forms of the format (largest value, the
subnormal step, the rounding error bound), and exactness where quantisation
loses nothing."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import fp8 as F


def test_every_code_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.e4m3_table()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.count_nonzero(np.isnan(ours)) == 2          # S.1111.111 only: no infinities


def test_format_closed_forms():
    t = F.e4m3_table()
    fin = t[~np.isnan(t)]
    assert fin.max() == 448.0 == F.E4M3_MAX               # the largest finite value the page gives
    pos = np.unique(fin[fin > 0])
    assert pos.min() == 2.0 ** -9                         # smallest subnormal: 2^-6 / 8
    assert 2.0 ** -6 in pos and 1.0 in pos                # smallest normal, one
    assert len(pos) == 126                                # 7 subnormals + 15 binades x 8 - 1 (NaN)
    # 3 mantissa bits: within a binade [2^e, 2^(e+1)) the values step by 2^(e-3)
    for e in range(-6, 8):
        vals = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert np.allclose(np.diff(vals), 2.0 ** (e - 3))


def test_encode_rounds_like_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x.astype(np.float64)), ref)
    # exact halfway points between neighbours: torch and the oracle both go to the even mantissa
    t = F.e4m3_table()[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)
    ref = torch.from_numpy(mids).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(mids.astype(np.float64)), ref)
    assert np.all(F.e4m3_encode(mids.astype(np.float64)) % 2 == 0)


def test_encode_saturates_and_keeps_sign_and_nan():
    assert F.e4m3_encode([1000.0, 449.0, 464.0, 1e30])[0] == 0x7E
    assert list(F.e4m3_encode([-1e30, -0.0, 0.0, math.nan])) == [0xFE, 0x80, 0x00, 0x7F]


def test_worked_example_5_7(golden):
    ex = golden["chapter5_example_5_7_fp8"]
    row = np.zeros(ex["row_length"])
    row[0], row[ex["block"]] = ex["first_elements"]
    # whole-row scale: max 10 maps to 448; the first element becomes 44.8, rounds to 44, comes back as 55/56
    sc = F.head_scale(row)
    codes = F.quantize_block(row, sc)
    assert F.e4m3_value(codes[0]) == ex["whole_row_scale"]["rounded_first"]
    tol = ex["tol_rel"]
    assert abs(F.e4m3_value(codes[0]) * float(sc) - 55 / 56) <= tol * 55 / 56
    assert abs(F.e4m3_value(codes[ex["block"]]) * float(sc) - 10.0) <= tol * 10.0
    # the first block's own scale (max 1): the element maps to 448 and comes back exactly
    sc1 = F.head_scale(row[:ex["block"]])
    c1 = F.quantize_block(row[:ex["block"]], sc1)
    assert F.e4m3_value(c1[0]) == ex["first_block_scale"]["scaled_first"]
    assert abs(F.e4m3_value(c1[0]) * float(sc1) - ex["first_block_scale"]["dequantised_first"]) <= tol


def test_quantisation_error_bound():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, 1, 512, 64))
    codes, sc = F.quantize_kv(x)
    deq = F.dequantize_kv(codes, sc)
    s = float(sc[0, 0])
    r = np.abs(x / s)
    err = np.abs(deq - x) / s
    normal = r >= 2.0 ** -6
    # half a mantissa step: 2^-4 relative in the normal range, 2^-10 absolute (in units of the scale) below
    assert np.all(err[normal] <= 2.0 ** -4 * r[normal] * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))
    assert np.abs(deq).max() == pytest.approx(np.abs(x).max(), rel=1e-6)   # amax maps onto 448 and back


def test_scales_are_per_head():
    x = np.zeros((2, 3, 4, 8))
    for b in range(2):
        for h in range(3):
            x[b, h, 1, 2] = (b + 1) * (h + 1) * 3.0
    x[1, 2] = 0.0
    _, sc = F.quantize_kv(x)
    for b in range(2):
        for h in range(3):
            want = np.float32(1.0) if (b, h) == (1, 2) else np.float32((b + 1) * (h + 1) * 3.0) / np.float32(448.0)
            assert sc[b, h] == want


def test_decode_fp8_is_exact_on_representable_caches():
    # codes chosen first; a head whose largest value is 448 * 2^k has scale exactly 2^k, so the
    # quantisation is lossless and the fp8 decode equals the plain decode of the same numbers
    rng = np.random.default_rng(7)
    B, Hq, Hkv, L, d = 2, 4, 2, 40, 16
    t = F.e4m3_table()
    fin = np.flatnonzero(~np.isnan(t))

    def cache(k):
        c = rng.choice(fin, size=(B, Hkv, L, d)).astype(np.uint8)
        c[:, :, 0, 0] = 0x7E                       # amax = 448 in every head
        return t[c] * 2.0 ** k

    kc, vc = cache(-7), cache(-5)
    q = rng.standard_normal((B, Hq, d))
    sl = np.array([L, 17])
    kcodes, ksc = F.quantize_kv(kc)
    vcodes, vsc = F.quantize_kv(vc)
    assert np.all(ksc == np.float32(2.0 ** -7)) and np.all(vsc == np.float32(2.0 ** -5))
    O8, L8 = F.decode_fp8(q, kcodes, vcodes, ksc, vsc, sl, 0.25)
    O, Lse = oracle.decode(q, kc, vc, sl, 0.25)
    assert np.array_equal(O8, O) and np.array_equal(L8, Lse)


def test_decode_fp8_close_to_bf16_decode_on_the_workload_shape():
    # information plus a loose sanity bound: E4M3 keys/values perturb O by a few per cent at most
    shp = W.DecodeShape("small", 2, 8, 2, 128, 64, 300, seed=11)
    q, kc, vc, sl = W.decode_inputs(shp)
    qd, kd, vd = W.to_f64(q), W.to_f64(kc), W.to_f64(vc)
    kcodes, ksc = F.quantize_kv(kd)
    vcodes, vsc = F.quantize_kv(vd)
    O8, _ = F.decode_fp8(qd, kcodes, vcodes, ksc, vsc, sl.numpy(), shp.scale)
    O, _ = oracle.decode(qd, kd, vd, sl.numpy(), shp.scale)
    assert np.abs(O8 - O).max() < 0.1
