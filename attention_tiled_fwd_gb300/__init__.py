"""Exact tiled attention on GB300: thin Python binding over libfa.so.

The functions here carry the C ABI's names (include/fa.h) and only marshal
arguments: they check tensor shapes and dtypes, allocate outputs with torch
when the caller passes none, hand raw device pointers and the current CUDA
stream to the library, and raise ``FAError`` on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; nothing falls
back to PyTorch or the CPU.

Layout: q, k, v, o, dO, dq, dk, dv are ``[B, H, N, D]`` contiguous CUDA
tensors; lse and delta are ``[B, H, N]`` float32.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _native
from ._native import FA_BF16, FA_F32, FAError

__all__ = ["fa_forward", "fa_backward_dq", "fa_backward_dkdv", "fa_backward_atomic", "fa_decode", "fa_decode_workspace_bytes",
           "fa_decode_noalloc",
           "fa_device_status", "fa_selftest_timeout", "FAError", "FA_BF16", "FA_F32", "attention_flops",
           "attention"]

_DT = {torch.bfloat16: FA_BF16, torch.float32: FA_F32}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16 or float32")
    return _DT[t.dtype]


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _shape4(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, D], got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return tuple(t.shape)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _scale(scale: Optional[float], D: int) -> float:
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def fa_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
               causal: bool = False, o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O = softmax(scale Q K^T) V and the natural log-sum-exp per row (fa_forward)."""
    shp = _shape4(q, "q")
    for t, n in ((k, "k"), (v, "v")):
        if _shape4(t, n) != shp or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    B, H, N, D = shp
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = _native.load()
    rc = lib.fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, _scale(scale, D),
                        int(bool(causal)), _dtype_code(q), _stream_ptr(stream))
    _native.check(rc, "fa_forward")
    return o, lse


def fa_backward_dq(q, k, v, o, dO, lse, scale: Optional[float] = None, causal: bool = False,
                   grad_dtype: torch.dtype = torch.float32, dq: Optional[torch.Tensor] = None,
                   delta: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """delta = rowsum(dO * O) and dQ (fa_backward_dq).  Returns (dq, delta)."""
    B, H, N, D = _shape4(q, "q")
    if dq is None:
        dq = torch.empty((B, H, N, D), dtype=grad_dtype, device=q.device)
    if delta is None:
        delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = _native.load()
    rc = lib.fa_backward_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta), _ptr(dq),
                            B, H, N, D, _scale(scale, D), int(bool(causal)), _dtype_code(q),
                            _dtype_code(dq), _stream_ptr(stream))
    _native.check(rc, "fa_backward_dq")
    return dq, delta


def fa_backward_dkdv(q, k, v, dO, lse, delta, scale: Optional[float] = None, causal: bool = False,
                     grad_dtype: torch.dtype = torch.float32, dk: Optional[torch.Tensor] = None,
                     dv: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """dK and dV (fa_backward_dkdv).  Returns (dk, dv)."""
    B, H, N, D = _shape4(q, "q")
    if dk is None:
        dk = torch.empty((B, H, N, D), dtype=grad_dtype, device=q.device)
    if dv is None:
        dv = torch.empty((B, H, N, D), dtype=grad_dtype, device=q.device)
    if dk.dtype != dv.dtype:
        raise ValueError("dk and dv must share a dtype")
    lib = _native.load()
    rc = lib.fa_backward_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(delta), _ptr(dk), _ptr(dv),
                              B, H, N, D, _scale(scale, D), int(bool(causal)), _dtype_code(q),
                              _dtype_code(dk), _stream_ptr(stream))
    _native.check(rc, "fa_backward_dkdv")
    return dk, dv


def fa_backward_atomic(q, k, v, o, dO, lse, scale: Optional[float] = None, causal: bool = False,
                       grad_dtype: torch.dtype = torch.float32, dq_accum: Optional[torch.Tensor] = None,
                       dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                       dv: Optional[torch.Tensor] = None, delta: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None):
    """The 5-GEMM comparator backward (fa_backward_atomic).  Returns (dq, dk, dv, delta).

    dq_accum is an fp32 CUDA tensor of at least B*H*N*D elements; outputs and dq_accum are
    allocated here when the caller passes none (dq, dk, dv in grad_dtype unless given)."""
    B, H, N, D = _shape4(q, "q")
    if dq is None:
        dq = torch.empty((B, H, N, D), dtype=grad_dtype, device=q.device)
    if dk is None:
        dk = torch.empty_like(dq)
    if dv is None:
        dv = torch.empty_like(dq)
    if not (dq.dtype == dk.dtype == dv.dtype):
        raise ValueError("dq, dk and dv must share a dtype")
    if delta is None:
        delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if dq_accum is None:
        dq_accum = torch.empty((B, H, N, D), dtype=torch.float32, device=q.device)
    lib = _native.load()
    rc = lib.fa_backward_atomic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(dq_accum), dq_accum.numel() * dq_accum.element_size(),
                                B, H, N, D, _scale(scale, D), int(bool(causal)), _dtype_code(q), _dtype_code(dq),
                                _stream_ptr(stream))
    _native.check(rc, "fa_backward_atomic")
    return dq, dk, dv, delta


def fa_decode_workspace_bytes(B: int, H: int, n_q: int, N: int, D: int) -> int:
    """Workspace bytes fa_decode needs (fa_decode_workspace_bytes)."""
    import ctypes
    out = ctypes.c_size_t(0)
    _native.check(_native.load().fa_decode_workspace_bytes(B, H, n_q, N, D, ctypes.byref(out)),
                  "fa_decode_workspace_bytes")
    return int(out.value)


def fa_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
              causal: bool = False, o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Decode: q [B, H, n_q, D] (the last n_q positions) against k, v [B, H, N, D] (fa_decode).

    The workspace is a CUDA uint8 tensor of at least fa_decode_workspace_bytes(...) bytes; one is
    allocated here when the caller passes none.  Returns (o, lse)."""
    B, H, nq, D = _shape4(q, "q")
    Bk, Hk, N, Dk = _shape4(k, "k")
    if (Bk, Hk, Dk) != (B, H, D) or _shape4(v, "v") != (B, H, N, D):
        raise ValueError("k and v must be [B, H, N, D] matching q's B, H, D")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, nq), dtype=torch.float32, device=q.device)
    need = fa_decode_workspace_bytes(B, H, nq, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    lib = _native.load()
    rc = lib.fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, nq, N, D, _scale(scale, D),
                       int(bool(causal)), _ptr(workspace), workspace.numel() * workspace.element_size(),
                       _stream_ptr(stream))
    _native.check(rc, "fa_decode")
    return o, lse


def fa_decode_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                      scale: Optional[float] = None, causal: bool = False,
                      stream: Optional[torch.cuda.Stream] = None):
    """fa_decode with no workspace (fa_decode_noalloc): the partials go to the library's fixed
    per-device scratch, so the call allocates nothing; the caller passes the outputs o
    [B, H, n_q, D] bf16 and lse [B, H, n_q] fp32.  Calls that overlap in time on one device race on
    that scratch; sizes needing more than FA_DECODE_NOALLOC_SCRATCH_BYTES raise FAError
    (FA_ERR_SCRATCH_LIMIT).  Returns (o, lse)."""
    B, H, nq, D = _shape4(q, "q")
    Bk, Hk, N, Dk = _shape4(k, "k")
    if (Bk, Hk, Dk) != (B, H, D) or _shape4(v, "v") != (B, H, N, D):
        raise ValueError("k and v must be [B, H, N, D] matching q's B, H, D")
    if _shape4(o, "o") != (B, H, nq, D) or tuple(lse.shape) != (B, H, nq):
        raise ValueError("o must be [B, H, n_q, D] and lse [B, H, n_q]")
    rc = _native.load().fa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, nq, N, D,
                                          _scale(scale, D), int(bool(causal)), _stream_ptr(stream))
    _native.check(rc, "fa_decode_noalloc")
    return o, lse


def fa_device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return _native.load().fa_device_status(_stream_ptr(stream))


def fa_selftest_timeout(limit_us: int, stream: Optional[torch.cuda.Stream] = None) -> None:
    _native.check(_native.load().fa_selftest_timeout(int(limit_us), _stream_ptr(stream)), "fa_selftest_timeout")


def attention_flops(B: int, H: int, N: int, D: int, causal: bool, pass_: str = "fwd") -> float:
    """Algorithmic FLOPs: forward 4 B H N^2 D (two N x N x D GEMMs); the split
    backward counted as its 7 GEMMs, 14 B H N^2 D; both halved when causal."""
    per = {"fwd": 4.0, "bwd": 14.0, "bwd_dq": 6.0, "bwd_dkdv": 8.0}[pass_]
    f = per * B * H * float(N) * N * D
    return f / 2 if causal else f


from .autograd import attention  # noqa: E402  (differentiable wrapper over the functions above)
