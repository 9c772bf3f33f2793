"""Parity of the prefill's split tail (attn_fwd_ws) with the float64 oracle.

A non-causal call whose work units leave the last round of persistent CTAs partly filled
splits those units along their key blocks, and a merge kernel combines the pieces. The
environment variable GB300_ATTN_PREFILL_CTAS caps the CTA count, so that small problems reach
the split; the policy is mirrored in `split_plan` to pick cases that do split, and the launch
counter confirms that the merge kernel ran. Rows outside the split units must be bitwise equal
to attn_fwd's (no workspace); the split rows agree with the oracle at the usual tolerances.
"""
import ctypes
import math

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


def units_of(B, Hq, Hkv, Tq):
    n_qt = (Tq + 127) // 128
    g = Hq // Hkv
    return n_qt * (Hq // 2) * B if g % 2 == 0 else (n_qt + 1) // 2 * Hq * B


def split_plan(B, Hq, Hkv, Tq, Tk, ctas, causal):
    """(grid, full units, pieces per split unit) as the launcher chooses them."""
    units = units_of(B, Hq, Hkv, Tq)
    grid = min(units, ctas)
    if causal or grid >= units:
        return grid, units, 1
    r = units % grid
    s = min(grid // r, (Tk + 127) // 128) if r else 1
    return (grid, units - r, s) if s >= 2 else (grid, units, 1)


def unit_rows(B, Hq, Hkv, Tq, unit):
    """(b, head, first row) of the two tiles of a unit, in the kernel's non-causal unit order:
    (batch, head) major, the row tile fastest."""
    n_qt = (Tq + 127) // 128
    g = Hq // Hkv
    if g % 2 == 0:
        rest, rank = divmod(unit, n_qt)
        b, hp = divmod(rest, Hq // 2)
        return [(b, 2 * hp, rank * 128), (b, 2 * hp + 1, rank * 128)]
    rest, rank = divmod(unit, (n_qt + 1) // 2)
    b, h = divmod(rest, Hq)
    return [(b, h, 2 * rank * 128), (b, h, (2 * rank + 1) * 128)]


def split_mask(B, Hq, Hkv, Tq, full_units):
    m = np.zeros((B, Hq, Tq), dtype=bool)
    for u in range(full_units, units_of(B, Hq, Hkv, Tq)):
        for b, h, r0 in unit_rows(B, Hq, Hkv, Tq, u):
            m[b, h, r0:min(r0 + 128, Tq)] = True
    return m


CASES = [
    # B, Hq, Hkv, Tq, Tk, d, ctas
    (1, 3, 3, 1000, 1000, 64, 5),     # MHA row-tile pairs, 12 units: 2 split in 2
    (1, 4, 2, 900, 900, 128, 7),      # head pairs, 16 units: 2 split in 3 (4 ragged rows each)
    (1, 4, 2, 1024, 1024, 128, 5),    # head pairs, 16 units: 1 split in 5, full tiles
    (2, 8, 2, 640, 1300, 64, 13),     # g = 4, 40 units: 1 split in 11 one-block pieces, ragged keys
    (1, 2, 2, 1100, 1100, 128, 4),    # 10 units; the split ones hold an inactive second tile
    (1, 2, 1, 300, 2000, 128, 2),     # Tq < Tk: 3 units, 1 split in 2 pieces of 8 blocks
    (3, 6, 2, 384, 700, 64, 8),       # g = 3 row tiles, 36 units: 4 split in 2
    (1, 2, 2, 5376, 2600, 64, 40),    # 42 units: 2 split in 20 (more pieces than one merge batch)
    (36, 1, 1, 256, 4480, 128, 35),   # 36 units: 1 split in 35 (more pieces than a warp's lanes)
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,ctas", CASES)
def test_split_tail_matches_oracle(attn, monkeypatch, B, Hq, Hkv, Tq, Tk, d, ctas):
    grid, full, s = split_plan(B, Hq, Hkv, Tq, Tk, ctas, False)
    assert s >= 2, "case must reach the split"
    monkeypatch.setenv("GB300_ATTN_PREFILL_CTAS", str(ctas))
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, Tq, Tk, d, 900 + ctas + d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    n0 = attn.kernel_launches()
    o, lse = attn.fwd(qd, kd, vd, causal=False, scale=scale)
    torch.cuda.synchronize()
    assert attn.kernel_launches() - n0 == 2, "forward + merge"
    assert attn.last_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), False, scale)
    assert_attn_close(o, lse, O, L, f"split B{B} Hq{Hq} Hkv{Hkv} Tq{Tq} Tk{Tk} d{d} ctas{ctas}")
    m = split_mask(B, Hq, Hkv, Tq, full)
    assert_attn_close(f64(o)[m], f64(lse)[m], O[m], L[m], "rows of the split units")

    # without a workspace the same CTAs run every unit whole: other rows are bitwise equal
    n0 = attn.kernel_launches()
    o1 = torch.empty_like(o)
    l1 = torch.empty_like(lse)
    st = attn.lib().attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), l1.data_ptr(), B, Hq, Hkv,
                             Tq, Tk, d, 0, scale, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert attn.kernel_launches() - n0 == 1
    keep = torch.from_numpy(~m).to(DEV)
    assert torch.equal(o[keep], o1[keep]) and torch.equal(lse[keep], l1[keep])


def test_split_tail_is_deterministic(attn, monkeypatch):
    monkeypatch.setenv("GB300_ATTN_PREFILL_CTAS", "13")
    q, k, v = W.attention_inputs_custom(2, 8, 2, 640, 1300, 64, 31)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = attn.fwd(qd, kd, vd, causal=False)
    o2, l2 = attn.fwd(qd, kd, vd, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_is_never_split(attn, monkeypatch):
    monkeypatch.setenv("GB300_ATTN_PREFILL_CTAS", "5")
    q, k, v = W.attention_inputs_custom(1, 3, 3, 1000, 1000, 64, 32)
    n0 = attn.kernel_launches()
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert attn.kernel_launches() - n0 == 1
    O, L = oracle.attention(f64(q), f64(k), f64(v), True, 1.0 / 8.0)
    assert_attn_close(o, lse, O, L, "causal, capped CTAs")


def test_workspace_arguments_are_checked(attn):
    lib = attn.lib()
    q, k, v = [t.to(DEV) for t in W.attention_inputs_custom(1, 2, 2, 256, 256, 64, 33)]
    o = torch.empty_like(q)
    need = attn.fwd_workspace_size(64)
    assert need == attn.fwd_workspace_size(64) > 0 and attn.fwd_workspace_size(96) == 0
    assert attn.fwd_workspace_size(128) > need
    ws = torch.empty(need + 64, dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream

    def call(ptr, nbytes):
        return lib.attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, 1, 2, 2, 256, 256, 64,
                               0, 0.125, ptr, ctypes.c_size_t(nbytes), s)

    assert call(None, 16) == 4                      # NULL with a size
    assert call(ws.data_ptr(), need - 1) == 4       # too small
    assert call(ws.data_ptr() + 8, need) == 3       # misaligned
    assert call(ws.data_ptr(), need) == 0
    assert call(None, 0) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("shape", [W.MHA_GPT2, W.AttnShape("non-causal MHA B1 H20 T4096 d128", 1, 20, 20, 4096, 128,
                                                           False, 3100)],
                         ids=["mha-b8-h12-d64", "mha-b1-h20-d128"])
def test_full_size_mha_tail_rows(attn, shape):
    """Non-causal MHA on every SM (B8 H12 T4096 d64: 1536 units, 16 in the last round; B1 H20
    T4096 d128: 320 units, 16 in the last round): the last round's units are split; their rows
    (all row tiles of the last head) against the oracle, and the rest bitwise equal to the
    unsplit kernel."""
    shp = shape
    q, k, v = W.attention_inputs(shp)[:3]
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    n0 = attn.kernel_launches()
    o, lse = attn.fwd(qd, kd, vd, causal=False, scale=shp.scale)
    torch.cuda.synchronize()
    split = attn.kernel_launches() - n0 == 2
    o1 = torch.empty_like(o)
    l1 = torch.empty_like(lse)
    assert attn.lib().attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), l1.data_ptr(), shp.B,
                               shp.Hq, shp.Hkv, shp.T, shp.T, shp.d, 0, shp.scale,
                               torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid, full, s = split_plan(shp.B, shp.Hq, shp.Hkv, shp.T, shp.T, sms, False)
    assert split == (s >= 2)
    m = split_mask(shp.B, shp.Hq, shp.Hkv, shp.T, full)
    keep = torch.from_numpy(~m).to(DEV)
    assert torch.equal(o[keep], o1[keep]) and torch.equal(lse[keep], l1[keep])
    if not split:
        return
    heads = sorted({(b, h) for b, h in zip(*np.nonzero(m.any(axis=2)))})
    rng = np.random.default_rng(5)
    O_all, L_all, o_all, l_all = [], [], [], []
    for b, h in heads[:: max(1, len(heads) // 6)] + [heads[-1]]:
        rows = np.nonzero(m[b, h])[0]
        edges = [r for r in (127, 128, 255, 256, 2047, 2048) if m[b, h, r]]  # tile and piece boundaries
        rows = np.unique(np.concatenate([rows[:2], rows[-2:], rng.choice(rows, 6), edges]).astype(np.int64))
        Or, Lr = oracle.attention_rows(f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h:h + 1]), f64(v[b:b + 1, h:h + 1]),
                                       0, 0, rows, False, shp.scale)
        O_all.append(Or)
        L_all.append(Lr)
        o_all.append(f64(o[b, h, rows]))
        l_all.append(f64(lse[b, h, rows]))
    assert_attn_close(np.concatenate(o_all), np.concatenate(l_all), np.concatenate(O_all), np.concatenate(L_all),
                      "split rows, full size")
