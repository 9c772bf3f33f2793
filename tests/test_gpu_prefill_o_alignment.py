"""The prefill's O stores: 32-byte stores when O is 32-byte aligned, 16-byte stores otherwise
(the C ABI only requires 16-byte alignment). An O buffer offset by 16 bytes from an aligned
allocation takes the second path; its result must be bitwise equal to the aligned call's and
agree with the float64 oracle."""
import math

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


@pytest.mark.parametrize("B,Hq,Hkv,T,d,causal", [(1, 4, 2, 700, 128, True), (2, 3, 3, 520, 64, False),
                                                 (1, 8, 2, 1024, 128, False)])
def test_o_offset_by_16_bytes(attn, B, Hq, Hkv, T, d, causal):
    q, k, v = W.attention_inputs_custom(B, Hq, Hkv, T, T, d, 4100 + d + T)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    o_al, l_al = attn.fwd(qd, kd, vd, causal=causal, scale=scale)
    flat = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=DEV)
    o_16 = flat[8:].view(q.shape)
    assert o_16.data_ptr() % 32 == 16 and o_al.data_ptr() % 32 == 0
    _, l_16 = attn.fwd(qd, kd, vd, causal=causal, scale=scale, out=o_16)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    assert torch.equal(o_16, o_al) and torch.equal(l_16, l_al)
    O, L = oracle.attention(f64(q), f64(k), f64(v), causal, scale)
    assert_attn_close(o_16, l_16, O, L, f"O offset by 16 bytes B{B} Hq{Hq} Hkv{Hkv} T{T} d{d} causal{causal}")
