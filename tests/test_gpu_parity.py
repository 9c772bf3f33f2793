"""Parity of the CUDA path (through the C ABI) with the float64 oracle at sizes
the oracle finishes in seconds: several tiles, ragged tails, the degenerate
cases, both head dims, every grouping mode of the prefill kernel, and the
split-count range of flash-decoding."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import assert_attn_close, assert_norm_close, bf16_round, f64, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


DEV = "cuda"


def _prefill_case(attn, B, Hq, Hkv, Tq, Tk, d, causal, seed, q_scale=1.0, scale=None):
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, seed, q_scale=q_scale)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    O, L = oracle.attention(f64(q), f64(k), f64(v), causal, scale)
    return o, lse, O, L


# ----------------------------------------------------------------------------- prefill

def test_single_head_workload_fp32_inputs(attn):
    # 1 x 1 x 256 x 64 causal, fp32 N(0,1) inputs rounded once to bf16
    shp = W.SINGLE_HEAD
    q, k, v, (q32, k32, v32) = W.attention_inputs(shp)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=shp.scale)
    torch.cuda.synchronize()
    O, L = oracle.attention(f64(q), f64(k), f64(v), True, shp.scale)
    assert_attn_close(o, lse, O, L, "single head")
    # information only: distance to the oracle on the unrounded fp32 inputs
    O32, _ = oracle.attention(f64(q32), f64(k32), f64(v32), True, shp.scale)
    print("max |O - O*(fp32 inputs)| =", np.abs(f64(o) - O32).max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (8, 2), (6, 2), (3, 1)])
def test_prefill_grouping_modes(attn, d, causal, Hq, Hkv):
    # g = 1, 2, 4 (pairs of heads) and g = 3 (pairs of row tiles); T spans 3 tiles + a ragged tail
    o, lse, O, L = _prefill_case(attn, 2, Hq, Hkv, 300, 300, d, causal, seed=100 + Hq + d)
    assert_attn_close(o, lse, O, L, f"B2 Hq{Hq} Hkv{Hkv} d{d} causal{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,T", [(16, 3, 3, 1100), (20, 4, 2, 640), (8, 5, 1, 1500)])
def test_prefill_persistent_schedule(attn, d, causal, B, Hq, Hkv, T):
    # More work units than SMs (240, 200, 240), so each persistent CTA walks several units of
    # different lengths; with g odd and an odd tile count (9 tiles of 1100 rows) the last row
    # pair of every head has an inactive second tile, first in the causal order, last otherwise.
    o, lse, O, L = _prefill_case(attn, B, Hq, Hkv, T, T, d, causal, seed=700 + Hq + d + T)
    assert_attn_close(o, lse, O, L, f"B{B} Hq{Hq} Hkv{Hkv} T{T} d{d} causal{causal}")


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 255, 256, 257, 640])
def test_prefill_lengths_and_tails(attn, T):
    for causal in (False, True):
        o, lse, O, L = _prefill_case(attn, 1, 2, 1, T, T, 128, causal, seed=200 + T)
        assert_attn_close(o, lse, O, L, f"T{T} causal{causal}")


@pytest.mark.parametrize("Tq,Tk", [(100, 300), (300, 100), (1, 513), (513, 1), (128, 384)])
def test_prefill_rectangular(attn, Tq, Tk):
    for causal in (False, True):
        o, lse, O, L = _prefill_case(attn, 1, 4, 2, Tq, Tk, 64, causal, seed=300 + Tq + Tk)
        assert_attn_close(o, lse, O, L, f"Tq{Tq} Tk{Tk} causal{causal}")


def test_prefill_single_key_returns_its_value(attn):
    o, lse, O, L = _prefill_case(attn, 1, 4, 4, 5, 1, 128, False, seed=5)
    assert_attn_close(o, lse, O, L, "Tk=1")
    q, k, v = W.attention_inputs_custom(1, 4, 4, 5, 1, 128, 5)
    # every row must return v_0 exactly (rounded to bf16, which v already is)
    assert torch.equal(o.cpu(), v.expand(1, 4, 5, 128))


def test_prefill_causal_row0_is_v0(attn):
    q, k, v = W.attention_inputs_custom(1, 4, 2, 256, 256, 128, 9)
    o, _ = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    vv = v.repeat_interleave(2, dim=1)
    assert torch.equal(o[:, :, 0].cpu(), vv[:, :, 0])


def test_prefill_constant_values(attn):
    q, k, _ = W.attention_inputs_custom(1, 2, 1, 300, 300, 64, 10)
    v = torch.full((1, 1, 300, 64), 0.8125, dtype=torch.bfloat16)
    o, _ = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    # P is rounded to bf16 for the P.V product while l sums the fp32 P, so the
    # constant comes back within one bf16 ulp (2^-8 at 0.8125), not bit-exactly
    assert (o.float().cpu() - 0.8125).abs().max() <= 2 ** -8


def test_prefill_zero_queries_mean_and_log_count(attn):
    q = torch.zeros(1, 2, 260, 128, dtype=torch.bfloat16)
    _, k, v = W.attention_inputs_custom(1, 2, 2, 260, 260, 128, 11)
    for causal in (False, True):
        o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
        torch.cuda.synchronize()
        n = np.arange(1, 261) if causal else np.full(260, 260)
        assert np.abs(f64(lse)[0] - np.log(n)[None, :]).max() <= 1e-3
        O, L = oracle.attention(f64(q), f64(k), f64(v), causal, 1 / math.sqrt(128))
        assert_attn_close(o, lse, O, L, f"zero q causal{causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_peaked_scores(attn, causal):
    # q scaled by 100: nearly one-hot rows, the max moves a lot between blocks
    o, lse, O, L = _prefill_case(attn, 1, 2, 1, 384, 384, 64, causal, seed=12, q_scale=100.0)
    assert_attn_close(o, lse, O, L, f"peaked causal{causal}")


def test_prefill_increasing_scores_force_rescales(attn):
    # keys grow along the sequence so every block raises the row maximum by a lot
    d, T = 64, 640
    q = torch.ones(1, 1, T, d, dtype=torch.bfloat16)
    k = (torch.arange(T, dtype=torch.float32)[:, None] / 16.0).expand(T, d).reshape(1, 1, T, d).to(torch.bfloat16)
    _, _, v = W.attention_inputs_custom(1, 1, 1, T, T, d, 13)
    scale = 1.0 / d
    for causal in (False, True):
        o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
        torch.cuda.synchronize()
        O, L = oracle.attention(f64(q), f64(k), f64(v), causal, scale)
        assert_attn_close(o, lse, O, L, f"rescale causal{causal}")


def test_prefill_custom_scale_and_no_lse(attn):
    q, k, v = W.attention_inputs_custom(2, 4, 4, 200, 200, 64, 14)
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=False, scale=0.37, return_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    O, _ = oracle.attention(f64(q), f64(k), f64(v), False, 0.37)
    assert_attn_close(o, None, O, None, "scale 0.37")


def test_prefill_does_not_touch_inputs_or_outside_output(attn):
    q, k, v = W.attention_inputs_custom(1, 2, 1, 200, 200, 128, 15)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    flat = torch.full((2 * 200 * 128 + 2 * 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = flat[4096:4096 + 2 * 200 * 128].view(1, 2, 200, 128)
    lse_flat = torch.full((400 + 2048,), 7.0, dtype=torch.float32, device=DEV)
    lse = lse_flat[1024:1424].view(1, 2, 200)
    attn.fwd(qd, kd, vd, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(flat[:4096] == 7.0) and torch.all(flat[4096 + 2 * 200 * 128:] == 7.0)
    assert torch.all(lse_flat[:1024] == 7.0) and torch.all(lse_flat[1424:] == 7.0)
    assert torch.equal(qd.cpu(), q) and torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)


def test_prefill_deterministic(attn):
    q, k, v = W.attention_inputs_custom(1, 4, 2, 700, 700, 128, 16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = attn.fwd(qd, kd, vd, causal=True)
    o2, l2 = attn.fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ----------------------------------------------------------------------------- decode

def _decode_case(attn, B, Hq, Hkv, d, Lcap, lens, splits, seed):
    shp = W.DecodeShape("t", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=lens)
    qd, kd, vd, sd = q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV)
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), shp.scale)
    outs = []
    for S in splits:
        o, lse = attn.decode(qd, kd, vd, sd, num_splits=S)
        torch.cuda.synchronize()
        assert_attn_close(o, lse, O, L, f"decode B{B} Hq{Hq} Hkv{Hkv} d{d} S{S}")
        outs.append((o, lse))
    return outs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (8, 1), (6, 2), (16, 2)])
def test_decode_groupings(attn, d, Hq, Hkv):
    _decode_case(attn, 3, Hq, Hkv, d, 300, [1, 77, 300], [1, 4, 19], seed=400 + Hq + d)


def test_decode_split_range_and_lengths(attn):
    lens = [1, 15, 16, 17, 31, 32, 33, 1000, 4095, 4096]
    Lcap = 4096
    _decode_case(attn, len(lens), 8, 2, 128, Lcap, lens, [1, 2, 3, 8, 64, 255, 256], seed=500)


def test_decode_equals_prefill_last_row(attn):
    # decode of the last token == row L-1 of causal prefill over the same keys
    L = 333
    q, k, v = W.attention_inputs_custom(1, 8, 2, L, L, 128, 17)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o_p, l_p = attn.fwd(qd, kd, vd, causal=True)
    sl = torch.tensor([L], dtype=torch.int32, device=DEV)
    o_d, l_d = attn.decode(qd[:, :, L - 1].contiguous(), kd, vd, sl, num_splits=5)
    torch.cuda.synchronize()
    assert np.abs(f64(o_p[:, :, L - 1]) - f64(o_d)).max() <= 2e-2
    assert np.abs(f64(l_p[:, :, L - 1]) - f64(l_d)).max() <= 1e-3


def test_decode_deterministic_for_fixed_splits(attn):
    shp = W.DecodeShape("t", 4, 8, 2, 128, 1, 2000, 18)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=[2000, 5, 999, 1500])
    args = (q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV))
    a = attn.decode(*args, num_splits=7)
    b = attn.decode(*args, num_splits=7)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_out_of_range_lengths_are_defined(attn):
    # precondition is 1 <= L <= Lcap; outside it the kernel clamps (<= 0: O = 0, LSE = -inf)
    shp = W.DecodeShape("t", 3, 4, 2, 64, 1, 64, 19)
    q, kc, vc, _ = W.decode_inputs(shp, seqlens=[64, 64, 64])
    sl = torch.tensor([0, -5, 500], dtype=torch.int32)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=2)
    torch.cuda.synchronize()
    assert torch.all(o[:2].cpu() == 0) and torch.all(torch.isneginf(lse[:2].cpu()))
    O, L = oracle.decode(f64(q[2:]), f64(kc[2:]), f64(vc[2:]), [64], shp.scale)
    assert_attn_close(o[2:], lse[2:], O, L, "clamped length")


# ----------------------------------------------------------------------------- FP8 (E4M3) KV cache

def _assert_codes_equal(got, want, what):
    got = got.cpu().numpy() if isinstance(got, torch.Tensor) else got
    bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
    assert bad.size == 0, f"{what}: {bad.size} codes differ, first at {bad[:5]}: {got.reshape(-1)[bad[:5]]} vs " \
                          f"{want.reshape(-1)[bad[:5]]}"


@pytest.mark.parametrize("d", [64, 128])
def test_kv_quantize_fp8_matches_oracle_bytes(attn, d):
    # heads of very different ranges: N(0,1), x 300 (codes near 448 after scaling), x 1e-3, an
    # all-zero head (scale 1), a head with one large outlier (most codes subnormal)
    gen = torch.Generator().manual_seed(900 + d)
    x = torch.randn((2, 3, 300, d), generator=gen)
    x[0, 1] *= 300.0
    x[0, 2] *= 1e-3
    x[1, 0] = 0.0
    x[1, 1, 7, 3] = 5000.0
    x = x.to(torch.bfloat16)
    codes, sc = attn.kv_quantize_fp8(x.to(DEV))
    torch.cuda.synchronize()
    want_codes, want_sc = oracle.quantize_kv(f64(x))
    assert np.array_equal(sc.cpu().numpy(), want_sc), (sc.cpu().numpy(), want_sc)
    _assert_codes_equal(codes, want_codes, f"d{d}")


def _decode_fp8_case(attn, B, Hq, Hkv, d, Lcap, lens, splits, seed):
    shp = W.DecodeShape("t", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=lens)
    kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
    vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
    okc, oks = oracle.quantize_kv(f64(kc))
    ovc, ovs = oracle.quantize_kv(f64(vc))
    O, L = oracle.decode_fp8(f64(q), okc, ovc, oks, ovs, sl.numpy(), shp.scale)
    for S in splits:
        o, lse = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=S)
        torch.cuda.synchronize()
        assert attn.last_device_error() == 0
        assert_attn_close(o, lse, O, L, f"fp8 decode B{B} Hq{Hq} Hkv{Hkv} d{d} S{S}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (8, 1), (6, 2)])
def test_decode_fp8_groupings(attn, d, Hq, Hkv):
    _decode_fp8_case(attn, 3, Hq, Hkv, d, 320, [1, 77, 320], [1, 4, 20], seed=950 + Hq + d)


def test_decode_fp8_lengths_and_splits(attn):
    lens = [1, 15, 16, 17, 33, 1000, 2048]
    _decode_fp8_case(attn, len(lens), 8, 2, 128, 2048, lens, [1, 3, 64, 128], seed=970)


def test_decode_fp8_equals_bf16_decode_on_lossless_cache(attn):
    # a cache whose values are E4M3 values times 2^-6 with a 448 * 2^-6 maximum in every head
    # quantises losslessly, so the FP8 path must agree with the bf16 path to the tolerance
    gen = torch.Generator().manual_seed(980)
    B, Hq, Hkv, d, L = 2, 8, 2, 128, 512
    table = torch.tensor(oracle.e4m3_table()[:0x7F], dtype=torch.float32)
    idx = torch.randint(0, 0x7F, (2, B, Hkv, L, d), generator=gen)
    sign = torch.where(torch.rand((2, B, Hkv, L, d), generator=gen) < 0.5, -1.0, 1.0)
    vals = table[idx] * sign * 2.0 ** -6
    vals[:, :, :, 0, 0] = 448.0 * 2.0 ** -6
    kc, vc = vals[0].to(torch.bfloat16), vals[1].to(torch.bfloat16)
    assert torch.equal(kc.float(), vals[0]) and torch.equal(vc.float(), vals[1])
    q = torch.randn((B, Hq, d), generator=gen).to(torch.bfloat16)
    sl = torch.tensor([L, 300], dtype=torch.int32)
    kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
    vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
    assert torch.all(ksc == 2.0 ** -6) and torch.all(vsc == 2.0 ** -6)
    o8, l8 = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=4)
    O, Lse = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), 1.0 / math.sqrt(d))
    torch.cuda.synchronize()
    assert_attn_close(o8, l8, O, Lse, "lossless fp8 cache")


def test_decode_and_prefill_replay_from_cuda_graphs(attn):
    # the calls are capture-safe: captured once into CUDA graphs (the decode combine is a
    # programmatic dependent of the split kernel), replays give the eager results bit for bit
    shp = W.DecodeShape("t", 4, 8, 2, 128, 1, 1024, 33)
    q, kc, vc, sl = [t.to(DEV) for t in W.decode_inputs(shp, seqlens=[1024, 5, 700, 333])]
    kq, ks = attn.kv_quantize_fp8(kc)
    vq, vs = attn.kv_quantize_fp8(vc)
    S = 6
    ws = torch.empty(attn.decode_workspace_size(4, 8, 128, S), dtype=torch.uint8, device=DEV)
    ws8 = torch.empty_like(ws)
    o_e, l_e = attn.decode(q, kc, vc, sl, num_splits=S, workspace=ws)
    o8_e, l8_e = attn.decode_fp8(q, kq, vq, ks, vs, sl, num_splits=S, workspace=ws8)
    pq, pk, pv = [t.to(DEV) for t in W.attention_inputs_custom(1, 4, 2, 300, 300, 128, 34)]
    po_e, pl_e = attn.fwd(pq, pk, pv, causal=True)
    o_g, l_g = torch.empty_like(o_e), torch.empty_like(l_e)
    o8_g, l8_g = torch.empty_like(o8_e), torch.empty_like(l8_e)
    po_g, pl_g = torch.empty_like(po_e), torch.empty_like(pl_e)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.decode(q, kc, vc, sl, num_splits=S, workspace=ws, out=o_g, lse=l_g)
        attn.decode_fp8(q, kq, vq, ks, vs, sl, num_splits=S, workspace=ws8, out=o8_g, lse=l8_g)
        attn.fwd(pq, pk, pv, causal=True, out=po_g, lse=pl_g)
    for _ in range(3):
        o_g.zero_()
        o8_g.zero_()
        po_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)
        assert torch.equal(o8_g, o8_e) and torch.equal(l8_g, l8_e)
        assert torch.equal(po_g, po_e) and torch.equal(pl_g, pl_e)
    assert attn.last_device_error() == 0


# ----------------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("T,D", [(1, 8), (37, 64), (300, 1000), (4096, 1024), (33, 4096), (5, 8192), (17, 2056)])
def test_rmsnorm_shapes(attn, T, D):
    gen = torch.Generator().manual_seed(T * 31 + D)
    x = torch.randn(T, D, generator=gen).to(torch.bfloat16)
    w = (0.5 + torch.rand(D, generator=gen)).to(torch.bfloat16)
    y = attn.rmsnorm(x.to(DEV), w.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    assert_norm_close(y, oracle.rmsnorm(f64(x), f64(w), 1e-6), f"T{T} D{D}")


def test_rmsnorm_workload_full(attn):
    x, w = W.norm_inputs(W.NORM_QWEN)
    xd = x.to(DEV)
    y = attn.rmsnorm(xd, w.to(DEV), eps=W.NORM_QWEN.eps)
    torch.cuda.synchronize()
    assert_norm_close(y, oracle.rmsnorm(f64(x), f64(w), W.NORM_QWEN.eps), "X[4096,1024]")
    assert torch.equal(xd.cpu(), x)


def test_rmsnorm_special_inputs(attn):
    D = 1024
    x = torch.zeros(4, D, dtype=torch.bfloat16)
    x[1] = 1.0
    x[2, 0] = 1000.0
    x[3] = 1e-3
    w = torch.ones(D, dtype=torch.bfloat16)
    y = attn.rmsnorm(x.to(DEV), w.to(DEV), eps=1e-6).cpu()
    assert torch.all(y[0] == 0)
    assert torch.all(torch.isfinite(y))
    assert_norm_close(y, oracle.rmsnorm(f64(x), f64(w), 1e-6), "special")
    # unit weight: per-row RMS of the output ~ 1
    gen = torch.Generator().manual_seed(3)
    xr = torch.randn(16, D, generator=gen).to(torch.bfloat16)
    yr = f64(attn.rmsnorm(xr.to(DEV), w.to(DEV), eps=1e-6))
    assert np.abs(np.sqrt((yr ** 2).mean(axis=1)) - 1).max() < 1e-2


@pytest.mark.parametrize("D", [1024, 4096, 8192, 1000, 64])
def test_rmsnorm_batch_invariant(attn, D):
    # the same rows normalised alone (one block per row), in a batch of 512 (same shape) and in
    # batches of 513 and 1030 (a warp per row) must agree bit for bit
    gen = torch.Generator().manual_seed(70 + D)
    x = (torch.randn(1030, D, generator=gen) * 3).to(torch.bfloat16).to(DEV)
    w = (torch.rand(D, generator=gen) + 0.5).to(torch.bfloat16).to(DEV)
    full = attn.rmsnorm(x, w, eps=1e-6)
    part = attn.rmsnorm(x[:513].contiguous(), w, eps=1e-6)
    small = attn.rmsnorm(x[:512].contiguous(), w, eps=1e-6)
    torch.cuda.synchronize()
    assert torch.equal(full[:513], part) and torch.equal(full[:512], small)
    for i in (0, 5, 511, 512, 1029):
        one = attn.rmsnorm(x[i:i + 1].contiguous(), w, eps=1e-6)
        assert torch.equal(one[0], full[i]), f"row {i} differs when normalised alone"
    assert_norm_close(full, oracle.rmsnorm(f64(x), f64(w), 1e-6), f"D{D}")


@pytest.mark.parametrize("T,D", [(1, 4096), (7, 1024), (600, 1024), (4096, 1024), (33, 8192), (300, 1000)])
def test_rmsnorm_residual(attn, T, D):
    gen = torch.Generator().manual_seed(80 + T + D)
    x = torch.randn(T, D, generator=gen).to(torch.bfloat16)
    r = (torch.randn(T, D, generator=gen) * 0.5).to(torch.bfloat16)
    w = (torch.rand(D, generator=gen) + 0.5).to(torch.bfloat16)
    y, h = attn.rmsnorm_residual(x.to(DEV), r.to(DEV), w.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    Y, H = oracle.rmsnorm_residual(f64(x), f64(r), f64(w), 1e-6)
    # h is the exact sum rounded once to bf16
    assert np.array_equal(f64(h), bf16_round(H))
    assert_norm_close(y, Y, f"residual T{T} D{D}")
    # in place: h written over r gives the same y and h
    rd = r.to(DEV)
    y2, h2 = attn.rmsnorm_residual(x.to(DEV), rd, w.to(DEV), eps=1e-6, h=rd)
    torch.cuda.synchronize()
    assert h2.data_ptr() == rd.data_ptr()
    assert torch.equal(y2, y) and torch.equal(rd, h)
    # the normalisation equals rmsnorm of the stored h, bit for bit (same fixed order)
    assert torch.equal(attn.rmsnorm(h, w.to(DEV), eps=1e-6), y)


# ----------------------------------------------------------------------------- failure path

def test_bounded_wait_reports_timeout_and_context_survives(attn):
    assert attn.last_device_error() == 0
    attn.selftest_wait_timeout(2000)
    assert attn.last_device_error() == 6  # ATTN_ERR_TIMEOUT
    assert attn.last_device_error() == 0  # cleared
    # the context still works afterwards
    x = torch.ones(8, 64, dtype=torch.bfloat16, device=DEV)
    y = attn.rmsnorm(x, torch.ones(64, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert torch.allclose(y.float().cpu(), torch.ones(8, 64), atol=1e-2)
