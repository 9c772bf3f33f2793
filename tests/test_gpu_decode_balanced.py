"""Parity of the balanced decode schedule (num_splits = 0) with the float64 oracle.

The balanced kernel divides the key stream of all (sequence, head block) segments into equal
ranges of 64-key tiles, one per persistent CTA; a segment that a range boundary cuts is
finished by the merge kernel from one partial per piece. The cases cover every grouping,
lengths of 0, 1 and around tile boundaries, fewer tiles than CTAs (so that some CTAs have
no range), one long segment cut into hundreds of pieces (more than one merge group of 32),
the E4M3 cache, CUDA-graph replay and the full decode workload.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import assert_attn_close, f64, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def attn():
    return require_gpu()


def _inputs(B, Hq, Hkv, d, Lcap, lens, seed):
    shp = W.DecodeShape("t", B, Hq, Hkv, d, 1, Lcap, seed)
    q, kc, vc, sl = W.decode_inputs(shp, seqlens=lens)
    return shp, q, kc, vc, sl


def _balanced_case(attn, B, Hq, Hkv, d, Lcap, lens, seed):
    shp, q, kc, vc, sl = _inputs(B, Hq, Hkv, d, Lcap, lens, seed)
    n0 = attn.kernel_launches()
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    assert attn.kernel_launches() - n0 == 2  # balanced kernel + merge
    assert attn.last_device_error() == 0
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), shp.scale)
    assert_attn_close(o, lse, O, L, f"balanced decode B{B} Hq{Hq} Hkv{Hkv} d{d} Lcap{Lcap}")
    return o, lse, O, L


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (8, 1), (6, 2), (16, 2), (3, 3)])
def test_balanced_groupings(attn, d, Hq, Hkv):
    # g = 4, 1, 8 (two head blocks), 3, 8, 1; lengths on both sides of tile boundaries
    _balanced_case(attn, 5, Hq, Hkv, d, 700, [1, 63, 64, 65, 700], seed=1100 + Hq + Hkv + d)


def test_balanced_lengths_out_of_range_and_empty(attn):
    # 0 and negative lengths give O = 0 and LSE = -inf; lengths past Lcap are clamped to Lcap
    lens = [0, 5, -3, 512, 10_000, 129]
    shp, q, kc, vc, sl = _inputs(len(lens), 8, 2, 128, 512, [max(0, min(x, 512)) for x in lens], 1120)
    sl_raw = torch.tensor(lens, dtype=torch.int32)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl_raw.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    o, lse = f64(o), f64(lse)
    for b in (0, 2):
        assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b]))
    keep = [1, 3, 4, 5]
    O, L = oracle.decode(f64(q[keep]), f64(kc[keep]), f64(vc[keep]), sl.numpy()[keep], shp.scale)
    assert_attn_close(o[keep], lse[keep], O, L, "balanced decode, clamped lengths")


def test_balanced_fewer_tiles_than_ctas(attn):
    # 3 sequences of <= 100 keys, 2 K/V heads: 8 tiles in all, so most CTAs have no range
    _balanced_case(attn, 3, 8, 2, 128, 100, [100, 1, 64], seed=1130)


def test_balanced_one_long_segment_cut_into_many_pieces(attn):
    # one segment of 32768 keys = 512 tiles over every CTA: the merge takes one partial per
    # CTA, more than one group of 32
    _balanced_case(attn, 1, 1, 1, 128, 32768, [32768], seed=1140)


def test_balanced_short_context_workload(attn):
    shp = W.DecodeShape("short context", 16, 32, 8, 128, 1024, 2048, 1004)
    q, kc, vc, sl = W.decode_inputs(shp)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    O, L = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), shp.scale)
    assert_attn_close(o, lse, O, L, "balanced decode, short context")


def test_balanced_is_deterministic_and_close_to_split(attn):
    shp, q, kc, vc, sl = _inputs(6, 16, 4, 128, 3000, [3000, 17, 2048, 1, 999, 1500], 1150)
    qd, kd, vd, sd = q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV)
    o1, l1 = attn.decode(qd, kd, vd, sd, num_splits=0)
    o2, l2 = attn.decode(qd, kd, vd, sd, num_splits=0)
    o3, l3 = attn.decode(qd, kd, vd, sd, num_splits=8)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1.float() - o3.float()).abs().max().item() <= 2e-2
    assert (l1 - l3).abs().max().item() <= 1e-3


def test_balanced_graph_replay(attn):
    shp, q, kc, vc, sl = _inputs(4, 8, 2, 128, 1024, [1024, 300, 1, 777], 1160)
    qd, kd, vd, sd = q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV)
    ws = torch.empty(attn.decode_workspace_size(4, 8, 128, 0), dtype=torch.uint8, device=DEV)
    o = torch.empty(4, 8, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(4, 8, dtype=torch.float32, device=DEV)
    attn.decode(qd, kd, vd, sd, num_splits=0, workspace=ws, out=o, lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            attn.decode(qd, kd, vd, sd, num_splits=0, workspace=ws, out=o, lse=lse, stream=s)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("d", [64, 128])
def test_balanced_fp8(attn, d):
    lens = [1, 64, 65, 900, 2048, 333]
    shp, q, kc, vc, sl = _inputs(len(lens), 8, 2, d, 2048, lens, 1170 + d)
    kcodes, ksc = attn.kv_quantize_fp8(kc.to(DEV))
    vcodes, vsc = attn.kv_quantize_fp8(vc.to(DEV))
    okc, oks = oracle.quantize_kv(f64(kc))
    ovc, ovs = oracle.quantize_kv(f64(vc))
    O, L = oracle.decode_fp8(f64(q), okc, ovc, oks, ovs, sl.numpy(), shp.scale)
    o, lse = attn.decode_fp8(q.to(DEV), kcodes, vcodes, ksc, vsc, sl.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    assert_attn_close(o, lse, O, L, f"balanced fp8 decode d{d}")


def test_balanced_full_size(attn):
    shp = W.DECODE_LLAMA
    q, kc, vc, sl = W.decode_inputs(shp)
    o, lse = attn.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), num_splits=0)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    o, lse = f64(o), f64(lse)
    O = np.empty_like(o)
    L = np.empty_like(lse)
    for b in range(shp.B):  # one sequence at a time keeps the float64 copies small
        Ob, Lb = oracle.decode(f64(q[b:b + 1]), f64(kc[b:b + 1]), f64(vc[b:b + 1]), sl[b:b + 1].numpy(), shp.scale)
        O[b], L[b] = Ob[0], Lb[0]
    assert_attn_close(o, lse, O, L, "balanced decode full size")
