"""The torch.autograd wrapper: forward and gradients against the float64
oracle, and that it refuses what the kernels do not support."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BF16, BF16_REL, TOL_LSE, assert_close, cuda_or_skip, to_np
from synthetic_inputs import make_qkv


def test_wrapper_is_exported():
    import attention_tiled_fwd_gb300 as fa
    assert callable(fa.attention)
    assert "attention" in fa.__all__


@pytest.mark.gpu
@pytest.mark.parametrize("shape,causal", [((1, 2, 200, 64), True), ((2, 1, 333, 128), False),
                                          ((1, 1, 257, 128), True), ((1, 1, 150, 96), True),
                                          ((1, 1, 140, 256), False), ((1, 2, 99, 192), True)])
def test_autograd_matches_oracle(shape, causal):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D = shape
    t = make_qkv(B, H, N, D, seed=4242 + N, dtype="bf16", with_dO=True)
    q, k, v = (t[n].to(dev).requires_grad_(True) for n in ("q", "k", "v"))
    o = fa.attention(q, k, v, causal=causal)
    o.backward(t["dO"].to(dev))
    scale = 1.0 / np.sqrt(D)
    ref = oracle.backward(t["q"], t["k"], t["v"], t["dO"], scale, causal)
    assert_close(to_np(o), ref["o"], TOL_BF16, BF16_REL, what="O")
    assert q.grad.dtype == torch.bfloat16
    for name, g in (("dq", q.grad), ("dk", k.grad), ("dv", v.grad)):
        assert_close(to_np(g), ref[name], TOL_BF16, BF16_REL, what=name)


@pytest.mark.gpu
def test_autograd_in_a_graph_with_other_ops():
    """Gradients flow through the wrapper inside a larger expression (a residual and a sum)."""
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    t = make_qkv(1, 2, 130, 64, seed=99, dtype="bf16")
    q, k, v = (t[n].to(dev).requires_grad_(True) for n in ("q", "k", "v"))
    loss = (fa.attention(q, k, v, causal=True).float() * 2.0 + q.float()).sum()
    loss.backward()
    dO = torch.full((1, 2, 130, 64), 2.0, dtype=torch.bfloat16)
    ref = oracle.backward(t["q"], t["k"], t["v"], dO, 1.0 / 8.0, True)
    assert_close(to_np(q.grad) - 1.0, ref["dq"], TOL_BF16, BF16_REL, what="dq (minus the residual's 1)")
    assert_close(to_np(v.grad), ref["dv"], TOL_BF16, BF16_REL, what="dv")
