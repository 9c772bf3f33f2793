"""attn_decode_noalloc: flash-decoding for callers that cannot allocate.

Some callers cannot hand attn_decode a workspace: their KV-cache pool already
owns (nearly) all device memory, they run under an allocator or budget that
forbids new allocations, or they must not call cudaMalloc/cudaFree in the
middle of a step. attn_decode_noalloc keeps the split partials in a fixed
32 MiB array inside the library instead. These tests check, through the C ABI:

* on two calls in a row that share the array, the result equals what
  attn_decode returns, and both equal the float64 oracle, at the tolerances of
  every other GPU test (max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3),
  for split counts and for the balanced schedule (num_splits = 0);
* a warmed-up call changes the device's free memory by zero bytes;
* requests whose partials would not fit are refused before anything runs, and
  the binding's default split count is lowered until they fit.

This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from exact_tiled_attention_attn_gb300 import _lib
from exact_tiled_attention_attn_gb300.build import build

O_MAX_ABS, O_MEAN_ABS, LSE_MAX_ABS = 2e-2, 2e-3, 1e-3
SCRATCH = 32 * 2 ** 20
FAKE = 0x10000  # non-null, 16-byte aligned, never dereferenced (the call is refused first)


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_refuses_partials_larger_than_the_fixed_array(lib):
    # 16 x 64 heads x 1024 splits x (128 + 2) x 4 bytes = 545 MB > 32 MiB
    B, Hq, Hkv, d, Lcap, S = 16, 64, 8, 128, 32768, 1024
    assert lib.attn_decode_workspace_size(B, Hq, d, S) > SCRATCH
    st = lib.attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, B, Hq, Hkv, d, Lcap, 0.088, S, None)
    assert st == 4  # ATTN_ERR_WORKSPACE, before anything touches the device


def test_default_split_count_fits_the_fixed_array(lib):
    import exact_tiled_attention_attn_gb300 as attn
    assert attn.NOALLOC_SCRATCH_BYTES == SCRATCH
    # 64 sequences x 64 heads at a 32768-token cache: the plain default (32 splits) needs
    # 68 MB of partials; the binding's default halves it until it fits
    B, Hq, Hkv, d, Lcap = 64, 64, 8, 128, 32768
    assert lib.attn_decode_workspace_size(B, Hq, d, attn.default_splits(B, Hkv, Lcap)) > SCRATCH
    s = attn.noalloc_splits(B, Hq, Hkv, d, Lcap)
    assert s >= 1 and lib.attn_decode_workspace_size(B, Hq, d, s) <= SCRATCH
    assert s == 1 or lib.attn_decode_workspace_size(B, Hq, d, 2 * s) > SCRATCH
    # shapes that already fit keep the plain default
    assert attn.noalloc_splits(16, 32, 8, 128, 32768) == attn.default_splits(16, 8, 32768)


def _inputs(torch, shape, lens, seed):
    dev = torch.device("cuda", 0)
    q, kc, vc, sl = W.decode_inputs(shape, seqlens=lens, seed=seed)
    host = (q, kc, vc, np.asarray(lens))
    return host, (q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev))


def _f64(t):
    import torch
    return t.detach().to("cpu").to(torch.float64).numpy()


def _close_to(o, lse, O, L, what):
    err = np.abs(_f64(o) - O)
    assert np.all(np.isfinite(_f64(o))), what
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, f"{what}: {err.max():.3e} {err.mean():.3e}"
    assert np.abs(_f64(lse) - L).max() <= LSE_MAX_ABS, what


def _run_pair(lib, torch, shape, lens, splits, seed):
    """attn_decode and attn_decode_noalloc on the same inputs; both against the oracle."""
    (qh, kh, vh, lh), (q, kc, vc, sl) = _inputs(torch, shape, lens, seed)
    B, Hq, d = q.shape
    Hkv, Lcap = kc.shape[1], kc.shape[2]
    ws_bytes = lib.attn_decode_workspace_size(B, Hq, d, splits)
    assert 0 < ws_bytes <= SCRATCH
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    o_ref = torch.empty_like(q)
    l_ref = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    o_na = torch.full_like(q, 3.0)
    l_na = torch.full((B, Hq), 3.0, dtype=torch.float32, device=q.device)
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
    O, L = oracle.decode(_f64(qh), _f64(kh), _f64(vh), lh, shape.scale)
    _close_to(o_na, l_na, O, L, "attn_decode_noalloc vs oracle")
    _close_to(o_ref, l_ref, O, L, "attn_decode vs oracle")


@pytest.mark.gpu
def test_matches_attn_decode_and_oracle_on_two_calls_in_a_row(lib):
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


@pytest.mark.gpu
def test_balanced_schedule_matches_attn_decode_and_oracle(lib):
    # num_splits = 0: the balanced schedule's partials and prefix sums also go to the array
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test needs a CUDA device")
    shape = W.DecodeShape("t", 16, 32, 8, 128, 1024, 4096, 2026)
    _run_pair(lib, torch, shape, W.decode_lengths(shape), 0, seed=2026)
    small = W.DecodeShape("t", 5, 8, 2, 64, 1, 300, 2027)
    _run_pair(lib, torch, small, [1, 150, 300, 64, 65], 0, seed=2027)


@pytest.mark.gpu
def test_a_call_allocates_no_device_memory(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test needs a CUDA device")
    shp = W.DecodeShape("t", 8, 32, 8, 128, 500, 3000, 2026)
    lens = W.decode_lengths(shp)
    (qh, kh, vh, lh), (q, kc, vc, sl) = _inputs(torch, shp, lens, 2026)
    B, Hq, d = q.shape
    Hkv, Lcap = kc.shape[1], kc.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), o.data_ptr(), lse.data_ptr(),
            B, Hq, Hkv, d, Lcap, shp.scale, 16, stream)
    # the first call on the device may load the library's device code (the module image
    # holds the 32 MiB array); every later call must leave the free memory unchanged
    assert lib.attn_decode_noalloc(*args) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert lib.attn_decode_noalloc(*args) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert lib.attn_last_device_error(stream) == 0
    O, L = oracle.decode(_f64(qh), _f64(kh), _f64(vh), lh, shp.scale)
    _close_to(o, lse, O, L, "attn_decode_noalloc vs oracle")


@pytest.mark.gpu
def test_binding_default_splits_on_a_large_batch(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test needs a CUDA device")
    import exact_tiled_attention_attn_gb300 as attn
    # 64 sequences x 64 query heads over a 16384-token cache: the plain default split count
    # (16) would need 34 MB of partials. The lengths stay short so the oracle is quick: the
    # first 1500 rows of each sequence get the seeded draws, the rest of the cache is zero
    # (never read: every length is <= 1500).
    Lcap, Lmax = 16384, 1500
    shp = W.DecodeShape("t", 64, 64, 8, 128, 1, Lmax, 2027)
    lens = W.decode_lengths(shp)
    (qh, kh, vh, lh), (q, kc_s, vc_s, sl) = _inputs(torch, shp, lens, 2027)
    kc = torch.zeros(64, 8, Lcap, 128, dtype=torch.bfloat16, device=q.device)
    vc = torch.zeros_like(kc)
    kc[:, :, :Lmax].copy_(kc_s)
    vc[:, :, :Lmax].copy_(vc_s)
    del kc_s, vc_s
    assert lib.attn_decode_workspace_size(64, 64, 128, attn.default_splits(64, 8, Lcap)) > SCRATCH
    o = torch.empty_like(q)
    lse = torch.empty(64, 64, dtype=torch.float32, device=q.device)
    attn.decode_noalloc(q, kc, vc, sl, out=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    O, L = oracle.decode(_f64(qh), _f64(kh), _f64(vh), lh, shp.scale)
    _close_to(o, lse, O, L, "default splits, 64 x 64 heads")
    with pytest.raises(TypeError):
        attn.decode_noalloc(q, kc, vc, sl)  # out is required: the binding allocates nothing
