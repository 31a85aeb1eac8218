"""Differentiable attention for PyTorch training code, built on the C ABI.

``attention(q, k, v, causal, scale)`` returns O = softmax(scale Q K^T) V and
records what the split backward needs: its ``backward`` runs fa_backward_dq
(delta = rowsum(dO * O) and dQ) and then fa_backward_dkdv (dK, dV) on the
current stream -- the training-step integration that the MLX port of
"Learning Metal with FlashAttention" lacks (its custom kernel has no
backward).  Inputs are ``[B, H, N, D]`` bf16 CUDA tensors, D any multiple of
8 up to 256; gradients come back in the inputs' dtype.  Nothing here computes attention:
every step runs in the library's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import fa_backward_dkdv, fa_backward_dq, fa_forward


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal: bool, scale: Optional[float]):
        q, k, v = (t.contiguous() for t in (q, k, v))
        o, lse = fa_forward(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse = ctx.saved_tensors
        dO = dO.to(q.dtype).contiguous()
        dq, delta = fa_backward_dq(q, k, v, o, dO, lse, scale=ctx.scale, causal=ctx.causal, grad_dtype=q.dtype)
        dk, dv = fa_backward_dkdv(q, k, v, dO, lse, delta, scale=ctx.scale, causal=ctx.causal,
                                  grad_dtype=q.dtype)
        return dq, dk, dv, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: Optional[float] = None) -> torch.Tensor:
    """O = softmax(scale Q K^T) V (scale defaults to 1/sqrt(D)), differentiable in q, k and v."""
    return _Attention.apply(q, k, v, bool(causal), scale)
