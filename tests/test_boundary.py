"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects invalid arguments before launching anything.
No call here reaches a kernel, so these run without a GPU."""
import ctypes
import os
import re

import pytest

from exact_tiled_attention_attn_gb300 import _lib
from exact_tiled_attention_attn_gb300.build import ROOT, build


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"defined"}


def test_header_and_binding_agree():
    declared = _declared_functions()
    assert declared == set(_lib.SIGNATURES), declared ^ set(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(0) == b"ok"


def test_workspace_size_formula(lib):
    assert lib.attn_decode_workspace_size(16, 32, 128, 64) == 16 * 32 * 64 * 130 * 4
    assert lib.attn_decode_workspace_size(0, 32, 128, 64) == 0
    assert lib.attn_decode_workspace_size(1, 1, 64, -1) == 0
    # num_splits = 0 is the balanced schedule: two partial slots of 4 heads x (d + 2) floats per
    # CTA, two CTAs per SM of the current device, then 1028 ints of prefix sums (0 with no device)
    ws = lib.attn_decode_workspace_size(1, 1, 64, 0)
    assert ws == 0 or (ws - 1028 * 4) % (2 * 2 * 4 * 66 * 4) == 0
    assert lib.attn_decode_workspace_size(1, 1, 96, 0) == 0


def test_default_splits_in_range(lib):
    for B, Hkv, L in [(16, 8, 32768), (1, 1, 16), (1, 1, 100000), (64, 8, 2048)]:
        s = lib.attn_decode_default_splits(B, Hkv, L)
        assert 1 <= s <= (L + 15) // 16


FAKE = 0x10000  # a non-null, 16-byte-aligned value that is never dereferenced


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=1, Tq=8, Tk=8, d=64,
             causal=0, scale=0.125, stream=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Tq"],
                        a["Tk"], a["d"], a["causal"], a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(B=0), 1), (dict(Tq=0), 1), (dict(Tk=-1), 1),
    (dict(Hq=3, Hkv=2), 1), (dict(scale=0.0), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1), (dict(causal=2), 1), (dict(d=96), 2), (dict(d=256), 2),
    (dict(q=FAKE + 8), 3), (dict(v=FAKE + 2), 3), (dict(lse=FAKE + 2), 3),
])
def test_fwd_rejects_invalid_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _dec(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, d=128, Lcap=256,
             scale=0.1, S=4, ws=FAKE, wsb=None, stream=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = lib.attn_decode_workspace_size(a["B"], a["Hq"], a["d"], max(a["S"], 1))
    return lib.attn_decode(a["q"], a["kc"], a["vc"], a["sl"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                           a["d"], a["Lcap"], a["scale"], a["S"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(sl=None), 1), (dict(Hq=6, Hkv=4), 1), (dict(S=-1), 1),
    (dict(S=0, B=1025), 2), (dict(S=0, B=1024, Hkv=8, Hq=16, Lcap=1 << 28), 2),
    (dict(S=17), 1), (dict(Lcap=0), 1), (dict(scale=-1.0), 1), (dict(d=80), 2),
    (dict(Hq=18, Hkv=2), 2), (dict(kc=FAKE + 4), 3), (dict(sl=FAKE + 2), 3),
    (dict(ws=None), 4), (dict(wsb=16), 4), (dict(ws=FAKE + 8), 3),
])
def test_decode_rejects_invalid_arguments(lib, kw, code):
    assert _dec(lib, **kw) == code


@pytest.mark.parametrize("args,code", [
    ((None, FAKE, FAKE, 4, 1024, 1e-6), 1), ((FAKE, FAKE, FAKE, 0, 1024, 1e-6), 1),
    ((FAKE, FAKE, FAKE, 4, 1020, 1e-6), 1), ((FAKE, FAKE, FAKE, 4, 1024, -1.0), 1),
    ((FAKE, FAKE, FAKE, 4, 16384, 1e-6), 2), ((FAKE + 4, FAKE, FAKE, 4, 1024, 1e-6), 3),
])
def test_rmsnorm_rejects_invalid_arguments(lib, args, code):
    assert lib.rmsnorm_fwd(*args, None) == code


def test_rmsnorm_supported_widths(lib):
    # D > 4096 must be a multiple of 64 (eight whole segments of 16-byte vectors)
    assert lib.rmsnorm_fwd(FAKE, FAKE, FAKE, 4, 4104, 1e-6, None) == 2
    assert lib.rmsnorm_fwd(FAKE, FAKE, FAKE, 4, 8200, 1e-6, None) == 2


@pytest.mark.parametrize("args,code", [
    ((None, FAKE, FAKE, FAKE, FAKE, 4, 1024, 1e-6), 1), ((FAKE, None, FAKE, FAKE, FAKE, 4, 1024, 1e-6), 1),
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 64, 4, 1024, 1e-6), 1),  # y aliases x
    ((FAKE, FAKE + 64, FAKE, FAKE + 128, FAKE + 128, 4, 1024, 1e-6), 1),  # y aliases h
    ((FAKE, FAKE + 64, FAKE, FAKE + 128, FAKE + 192, 4, 4104, 1e-6), 2),
    ((FAKE, FAKE + 72, FAKE, FAKE + 128, FAKE + 192, 4, 1024, 1e-6), 3),
])
def test_rmsnorm_residual_rejects_invalid_arguments(lib, args, code):
    assert lib.rmsnorm_residual_fwd(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((None, FAKE, FAKE, 2, 4, 64, 128), 1), ((FAKE, FAKE, FAKE, 0, 4, 64, 128), 1),
    ((FAKE, FAKE, FAKE, 2, 4, 64, 12), 2), ((FAKE, FAKE, FAKE, 300, 300, 64, 128), 2),
    ((FAKE + 8, FAKE, FAKE, 2, 4, 64, 128), 3), ((FAKE, FAKE + 4, FAKE, 2, 4, 64, 128), 3),
])
def test_kv_quantize_rejects_invalid_arguments(lib, args, code):
    assert lib.attn_kv_quantize_fp8(*args, None) == code


def test_decode_fp8_needs_scales(lib):
    args = [FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 256, 0.1, 2, FAKE, 1 << 20, None]
    assert lib.attn_decode_fp8(*args) == 1
    args[3], args[4] = FAKE, FAKE + 2
    assert lib.attn_decode_fp8(*args) == 3


def _bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, Hq=4, Hkv=2,
             Tq=300, Tk=300, d=128, causal=1, scale=0.1, ws=FAKE, wsb=None, stream=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = lib.attn_bwd_workspace_size(a["B"], a["Hq"], a["Tq"])
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["B"],
                        a["Hq"], a["Hkv"], a["Tq"], a["Tk"], a["d"], a["causal"], a["scale"], a["ws"], a["wsb"],
                        a["stream"])


def test_bwd_workspace_size(lib):
    assert lib.attn_bwd_workspace_size(2, 32, 8192) == 2 * 32 * 8192 * 4
    assert lib.attn_bwd_workspace_size(1, 1, 3) == 256  # rounded up to 256 bytes
    assert lib.attn_bwd_workspace_size(0, 1, 3) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(do=None), 1), (dict(dv=None), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(Tk=0), 1), (dict(scale=0.0), 1), (dict(causal=2), 1), (dict(d=96), 2), (dict(dk=FAKE + 8), 3),
    (dict(lse=FAKE + 2), 3), (dict(ws=None), 4), (dict(wsb=16), 4), (dict(ws=FAKE + 8), 3),
])
def test_bwd_rejects_invalid_arguments(lib, kw, code):
    n0 = lib.attn_kernel_launches()
    assert _bwd(lib, **kw) == code
    assert lib.attn_kernel_launches() == n0


def test_selftest_rejects_out_of_range_bound(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == 1
    assert lib.attn_selftest_wait_timeout(2_000_000, None) == 1


def test_rejected_calls_launch_nothing(lib):
    n0 = lib.attn_kernel_launches()
    _fwd(lib, d=96)
    _dec(lib, S=0)
    lib.rmsnorm_fwd(None, FAKE, FAKE, 4, 1024, 1e-6, None)
    assert lib.attn_kernel_launches() == n0


def test_binding_refuses_cpu_tensors():
    import torch
    import exact_tiled_attention_attn_gb300 as attn
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        attn.rmsnorm(x, torch.ones(64, dtype=torch.bfloat16))
