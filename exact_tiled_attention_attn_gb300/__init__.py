"""Exact tiled attention, flash-decoding and fused RMSNorm for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libgb300attn.so`` (``include/attn.h``).
The binding only checks and marshals arguments (torch tensors -> device
pointers, the current CUDA stream); every step of the computation runs in the
library's CUDA kernels. PyTorch provides device memory and streams.

    o, lse = fwd(q, k, v, causal=True)             # q [B,Hq,T,d], k/v [B,Hkv,T,d], bf16
    dq, dk, dv = bwd(q, k, v, o, lse, do, causal=True)
    o, lse = decode(q, kcache, vcache, seqlens)     # q [B,Hq,d], caches [B,Hkv,Lcap,d]
    y = rmsnorm(x, w, eps=1e-6)                     # x [T,D], w [D]
    codes, sc = kv_quantize_fp8(kcache)             # E4M3 codes (uint8) + fp32 scale per (b, head)
    o, lse = decode_fp8(q, kcodes, vcodes, ksc, vsc, seqlens)
"""
from __future__ import annotations

import math

import torch

from . import _lib
from ._lib import AttnError  # noqa: F401

__all__ = ["fwd", "fwd_workspace_size", "bwd", "decode", "decode_noalloc", "noalloc_splits", "NOALLOC_SCRATCH_BYTES", "decode_fp8", "kv_quantize_fp8", "rmsnorm", "rmsnorm_residual",
           "decode_workspace_size",
           "default_splits",
           "last_device_error", "kernel_launches", "selftest_wait_timeout", "AttnError", "lib"]


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    return _lib.load()


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_tensor(name, t, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fwd_workspace_size(d: int) -> int:
    return int(_lib.load().attn_fwd_workspace_size(d))


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
        return_lse: bool = True, stream=None, workspace=None):
    """Exact attention O = softmax(scale * Q K^T + mask) V (bf16 in/out), and the fp32 LSE.

    q [B, Hq, Tq, d], k/v [B, Hkv, Tk, d], contiguous bf16 on one CUDA device.
    A non-causal call takes a scratch ``workspace`` (uint8 tensor of at least
    ``fwd_workspace_size(d)`` bytes; allocated when not given) that lets the library
    balance its last round of work; causal calls need none.
    """
    _check_tensor("q", q, torch.bfloat16, 4)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must both be [B, Hkv, Tk, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor("out", out, torch.bfloat16, 4)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    if workspace is None and not causal and d in (64, 128):
        workspace = torch.empty(fwd_workspace_size(d), dtype=torch.uint8, device=q.device)
        if stream is not None:
            workspace.record_stream(stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.load().attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None,
                                 B, Hq, Hkv, Tq, Tk, d, 1 if causal else 0, float(scale), ws_ptr, ws_bytes,
                                 _stream_ptr(stream))
    _lib.check("attn_fwd_ws", st)
    return out, lse


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """Gradients (dq, dk, dv) of fwd's output with respect to q, k, v, given the upstream
    gradient dout and the forward's o and lse (recomputation; bf16 in and out)."""
    _check_tensor("q", q, torch.bfloat16, 4)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("o", o, torch.bfloat16, 4)
    _check_tensor("dout", dout, torch.bfloat16, 4)
    _check_tensor("lse", lse, torch.float32, 3)
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must both be [B, Hkv, Tk, d] matching q")
    if o.shape != q.shape or dout.shape != q.shape or tuple(lse.shape) != (B, Hq, Tq):
        raise ValueError("o and dout must match q, lse must be [B, Hq, Tq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(_lib.load().attn_bwd_workspace_size(B, Hq, Tq))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = _lib.load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Tq, Tk, d,
                              1 if causal else 0, float(scale), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _lib.check("attn_bwd", st)
    return dq, dk, dv


def decode_workspace_size(B: int, Hq: int, d: int, num_splits: int) -> int:
    return int(_lib.load().attn_decode_workspace_size(B, Hq, d, num_splits))


def default_splits(B: int, Hkv: int, Lcap: int) -> int:
    return int(_lib.load().attn_decode_default_splits(B, Hkv, Lcap))


def decode(q, kcache, vcache, seqlens, scale: float | None = None, num_splits: int | None = None,
           workspace=None, out=None, lse=None, return_lse: bool = True, stream=None):
    """Flash-decoding: one query per sequence against a bf16 KV cache.

    q [B, Hq, d]; kcache/vcache [B, Hkv, Lcap, d]; seqlens int32 [B] on the device.
    ``workspace`` (uint8 tensor) is allocated when not given.
    """
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("kcache", kcache, torch.bfloat16, 4)
    _check_tensor("vcache", vcache, torch.bfloat16, 4)
    _check_tensor("seqlens", seqlens, torch.int32, 1)
    B, Hq, d = q.shape
    Hkv, Lcap = kcache.shape[1], kcache.shape[2]
    if kcache.shape != vcache.shape or kcache.shape[0] != B or kcache.shape[3] != d:
        raise ValueError("kcache and vcache must both be [B, Hkv, Lcap, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        num_splits = default_splits(B, Hkv, Lcap)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = _lib.load().attn_decode(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), seqlens.data_ptr(),
                                 out.data_ptr(), lse.data_ptr() if lse is not None else None,
                                 B, Hq, Hkv, d, Lcap, float(scale), int(num_splits),
                                 workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream))
    _lib.check("attn_decode", st)
    return out, lse


# Size of the library's fixed device array that holds attn_decode_noalloc's split
# partials (the limit include/attn.h states for that entry point).
NOALLOC_SCRATCH_BYTES = 32 << 20


def noalloc_splits(B: int, Hq: int, Hkv: int, d: int, Lcap: int) -> int:
    """The default split count, lowered (halved) until the partials fit the fixed array."""
    s = default_splits(B, Hkv, Lcap)
    while s > 1 and decode_workspace_size(B, Hq, d, s) > NOALLOC_SCRATCH_BYTES:
        s //= 2
    return s


def decode_noalloc(q, kcache, vcache, seqlens, out, lse=None, scale: float | None = None,
                   num_splits: int | None = None, stream=None):
    """``decode`` without a workspace, for callers that cannot allocate device memory
    at decode time (a KV-cache pool that owns the memory, an allocation budget, no
    allocation allowed mid-step). The split partials go to the library's fixed
    32 MiB device array, and this function allocates nothing either: the caller
    passes ``out`` [B, Hq, d] bf16 and, if it wants the LSE, ``lse`` [B, Hq] fp32
    (``lse=None`` skips writing it).

    ``num_splits=None`` takes the default split count, halved until the partials
    fit in 32 MiB. All such calls share the one array: calls that can overlap on
    the GPU must be serialised by the caller. The first call on a device looks the
    array up and should come before any stream capture. Raises AttnError
    (ATTN_ERR_WORKSPACE) when an explicit ``num_splits`` needs more than 32 MiB.
    Returns ``(out, lse)``.
    """
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("kcache", kcache, torch.bfloat16, 4)
    _check_tensor("vcache", vcache, torch.bfloat16, 4)
    _check_tensor("seqlens", seqlens, torch.int32, 1)
    _check_tensor("out", out, torch.bfloat16, 3)
    B, Hq, d = q.shape
    Hkv, Lcap = kcache.shape[1], kcache.shape[2]
    if kcache.shape != vcache.shape or kcache.shape[0] != B or kcache.shape[3] != d:
        raise ValueError("kcache and vcache must both be [B, Hkv, Lcap, d] matching q")
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 2)
        if tuple(lse.shape) != (B, Hq):
            raise ValueError("lse must be [B, Hq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        num_splits = noalloc_splits(B, Hq, Hkv, d, Lcap)
    st = _lib.load().attn_decode_noalloc(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), seqlens.data_ptr(),
                                         out.data_ptr(), lse.data_ptr() if lse is not None else None,
                                         B, Hq, Hkv, d, Lcap, float(scale), int(num_splits), _stream_ptr(stream))
    _lib.check("attn_decode_noalloc", st)
    return out, lse


def kv_quantize_fp8(x, codes=None, scale=None, stream=None):
    """E4M3 codes of a bf16 cache x [B, H, L, d] with one fp32 scale per (b, h):
    scale = amax / 448, code = RNE(x / scale) saturated at 448. Returns (codes uint8, scale)."""
    _check_tensor("x", x, torch.bfloat16, 4)
    B, H, L, d = x.shape
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    else:
        _check_tensor("codes", codes, torch.uint8, 4)
        if codes.shape != x.shape:
            raise ValueError("codes must have the shape of x")
    if scale is None:
        scale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    else:
        _check_tensor("scale", scale, torch.float32, 2)
        if tuple(scale.shape) != (B, H):
            raise ValueError("scale must be [B, H]")
    st = _lib.load().attn_kv_quantize_fp8(x.data_ptr(), codes.data_ptr(), scale.data_ptr(), B, H, L, d,
                                          _stream_ptr(stream))
    _lib.check("attn_kv_quantize_fp8", st)
    return codes, scale


def decode_fp8(q, kcodes, vcodes, k_scale, v_scale, seqlens, scale: float | None = None,
               num_splits: int | None = None, workspace=None, out=None, lse=None, return_lse: bool = True,
               stream=None):
    """Flash-decoding over an E4M3 KV cache (uint8 codes [B, Hkv, Lcap, d] and fp32
    scales [B, Hkv], e.g. from kv_quantize_fp8), dequantised in registers."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("kcodes", kcodes, torch.uint8, 4)
    _check_tensor("vcodes", vcodes, torch.uint8, 4)
    _check_tensor("k_scale", k_scale, torch.float32, 2)
    _check_tensor("v_scale", v_scale, torch.float32, 2)
    _check_tensor("seqlens", seqlens, torch.int32, 1)
    B, Hq, d = q.shape
    Hkv, Lcap = kcodes.shape[1], kcodes.shape[2]
    if kcodes.shape != vcodes.shape or kcodes.shape[0] != B or kcodes.shape[3] != d:
        raise ValueError("kcodes and vcodes must both be [B, Hkv, Lcap, d] matching q")
    if tuple(k_scale.shape) != (B, Hkv) or tuple(v_scale.shape) != (B, Hkv):
        raise ValueError("k_scale and v_scale must be [B, Hkv]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        num_splits = default_splits(B, Hkv, Lcap)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = _lib.load().attn_decode_fp8(q.data_ptr(), kcodes.data_ptr(), vcodes.data_ptr(), k_scale.data_ptr(),
                                     v_scale.data_ptr(), seqlens.data_ptr(), out.data_ptr(),
                                     lse.data_ptr() if lse is not None else None, B, Hq, Hkv, d, Lcap, float(scale),
                                     int(num_splits), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _lib.check("attn_decode_fp8", st)
    return out, lse


def rmsnorm(x, w, eps: float = 1e-6, out=None, stream=None):
    """Fused RMSNorm y = x / sqrt(mean(x^2) + eps) * w over the last axis; bf16 in/out."""
    _check_tensor("x", x, torch.bfloat16, 2)
    _check_tensor("w", w, torch.bfloat16, 1)
    T, D = x.shape
    if w.shape[0] != D:
        raise ValueError("w must have D elements")
    if out is None:
        out = torch.empty_like(x)
    st = _lib.load().rmsnorm_fwd(x.data_ptr(), w.data_ptr(), out.data_ptr(), T, D, float(eps),
                                 _stream_ptr(stream))
    _lib.check("rmsnorm_fwd", st)
    return out


def rmsnorm_residual(x, r, w, eps: float = 1e-6, out=None, h=None, stream=None):
    """h = bf16(x + r) and y = RMSNorm(h) * w in one pass; returns (y, h).
    ``h`` may be ``x`` or ``r`` (in-place update of the residual stream)."""
    _check_tensor("x", x, torch.bfloat16, 2)
    _check_tensor("r", r, torch.bfloat16, 2)
    _check_tensor("w", w, torch.bfloat16, 1)
    T, D = x.shape
    if r.shape != x.shape or w.shape[0] != D:
        raise ValueError("r must match x and w must have D elements")
    if out is None:
        out = torch.empty_like(x)
    if h is None:
        h = torch.empty_like(x)
    st = _lib.load().rmsnorm_residual_fwd(x.data_ptr(), r.data_ptr(), w.data_ptr(), out.data_ptr(), h.data_ptr(),
                                          T, D, float(eps), _stream_ptr(stream))
    _lib.check("rmsnorm_residual_fwd", st)
    return out, h


def last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status code."""
    return int(_lib.load().attn_last_device_error(_stream_ptr(stream)))


def kernel_launches() -> int:
    return int(_lib.load().attn_kernel_launches())


def selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    _lib.check("attn_selftest_wait_timeout",
               _lib.load().attn_selftest_wait_timeout(int(timeout_us), _stream_ptr(stream)))
