"""attn_decode_noalloc: flash-decoding for callers that cannot allocate.

Some callers cannot hand attn_decode a workspace: their KV-cache pool already
owns (nearly) all device memory, they run under an allocator or budget that
forbids new allocations, or they must not call cudaMalloc/cudaFree in the
middle of a step. attn_decode_noalloc keeps the split partials in a fixed
32 MiB array inside the library instead. These tests check, through the C ABI,
that it returns what attn_decode returns (same tolerance as every other GPU
test: max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3) on two calls in
a row that share the array, and that it refuses requests that would not fit.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from exact_tiled_attention_attn_gb300 import _lib
from exact_tiled_attention_attn_gb300.build import build

O_MAX_ABS, O_MEAN_ABS, LSE_MAX_ABS = 2e-2, 2e-3, 1e-3
FAKE = 0x10000  # non-null, 16-byte aligned, never dereferenced (the call is refused first)


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_refuses_partials_larger_than_the_fixed_array(lib):
    # 16 x 64 heads x 1024 splits x (128 + 2) x 4 bytes = 545 MB > 32 MiB
    B, Hq, Hkv, d, Lcap, S = 16, 64, 8, 128, 32768, 1024
    assert lib.attn_decode_workspace_size(B, Hq, d, S) > 32 * 2 ** 20
    st = lib.attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, B, Hq, Hkv, d, Lcap, 0.088, S, None)
    assert st == 4  # ATTN_ERR_WORKSPACE, before anything touches the device


def _run_pair(lib, torch, shape, lens, splits, seed):
    dev = torch.device("cuda", 0)
    q, kc, vc, sl = W.decode_inputs(shape, seqlens=lens, seed=seed)
    q, kc, vc, sl = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    B, Hq, d = q.shape
    Hkv, Lcap = kc.shape[1], kc.shape[2]
    ws_bytes = lib.attn_decode_workspace_size(B, Hq, d, splits)
    assert 0 < ws_bytes <= 32 * 2 ** 20
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o_ref = torch.empty_like(q)
    l_ref = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    o_na = torch.full_like(q, 3.0)
    l_na = torch.full((B, Hq), 3.0, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.attn_decode(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), o_ref.data_ptr(),
                         l_ref.data_ptr(), B, Hq, Hkv, d, Lcap, shape.scale, splits, ws.data_ptr(), ws_bytes, stream)
    assert st == 0
    st = lib.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), o_na.data_ptr(),
                                 l_na.data_ptr(), B, Hq, Hkv, d, Lcap, shape.scale, splits, stream)
    assert st == 0
    torch.cuda.synchronize()
    assert lib.attn_last_device_error(stream) == 0
    err = (o_na.float() - o_ref.float()).abs()
    assert torch.isfinite(o_na.float()).all()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    assert (l_na - l_ref).abs().max().item() <= LSE_MAX_ABS


@pytest.mark.gpu
def test_matches_attn_decode_on_two_calls_in_a_row(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test needs a CUDA device")
    # first call: 16 sequences x 32 heads x 64 splits x 130 floats = 17 MB of partials
    big = W.DecodeShape("t", 16, 32, 8, 128, 1024, 4096, 2024)
    lens = W.decode_lengths(big)
    _run_pair(lib, torch, big, lens, 64, seed=2024)
    # second call right after, other shape and lengths: the array still holds the
    # first call's partials, which must not leak into this result
    small = W.DecodeShape("t", 3, 8, 2, 64, 1, 300, 2025)
    _run_pair(lib, torch, small, [1, 150, 300], 7, seed=2025)
