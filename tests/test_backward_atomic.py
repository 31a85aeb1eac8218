"""The 5-GEMM comparator backward (fa_backward_atomic: dQ accumulated across
key tiles by L2 reduce-adds) vs the float64 oracle, through the C ABI, and its
argument checks."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_tiled_fwd_gb300 import _native as nat
from helpers import TOL_BF16, BF16_REL, assert_close, cuda_or_skip, to_np
from synthetic_inputs import make_qkv, sample_rows


@pytest.fixture(scope="module")
def lib():
    from attention_tiled_fwd_gb300 import build
    build.build()
    return nat.load()


def _call(lib, D=128, dtype=nat.FA_BF16, grad=nat.FA_BF16, ws_bytes=1 << 30, ptr=4096):
    p = ptr
    return lib.fa_backward_atomic(p, p, p, p, p, p, p, p, p, p, p, ws_bytes, 1, 1, 64, D, 0.1, 1, dtype, grad, None)


def test_rejects_before_touching_memory(lib):
    # checks that need no GPU: head dimension, dtype, shape, null pointers
    assert _call(lib, D=64) == nat.FA_ERR_HEAD_DIM
    assert _call(lib, D=256) == nat.FA_ERR_HEAD_DIM
    assert _call(lib, dtype=nat.FA_F32) == nat.FA_ERR_DTYPE
    assert _call(lib, grad=9) == nat.FA_ERR_DTYPE
    assert _call(lib, ptr=0) == nat.FA_ERR_NULL
    assert lib.fa_backward_atomic(*([4096] * 11), 1 << 30, 0, 1, 64, 128, 0.1, 1, 1, 1, None) == nat.FA_ERR_SHAPE


def _run(inp, causal, dev, scale, grad_dtype):
    import attention_tiled_fwd_gb300 as fa
    q, k, v, dO = (inp[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal)
    acc = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)  # must be cleared by the call
    dq, dk, dv, delta = fa.fa_backward_atomic(q, k, v, o, dO, lse, scale=scale, causal=causal,
                                              grad_dtype=grad_dtype, dq_accum=acc)
    assert fa.fa_device_status() == 0
    return dict(o=o, dq=dq, dk=dk, dv=dv, delta=delta)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 1, 1, 128), (1, 2, 77, 128), (2, 1, 300, 128), (1, 1, 640, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_atomic_backward_matches_oracle(shape, causal, grad_dtype):
    dev = cuda_or_skip()
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=700 + N, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    g = _run(inp, causal, dev, scale, grad_dtype)
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], scale, causal)
    rel = BF16_REL if grad_dtype == torch.bfloat16 else 0.0
    for n in ("dq", "dk", "dv"):
        assert_close(to_np(g[n]), ref[n], TOL_BF16, rel, what=f"{n} {shape} causal={causal}")
    # delta is formed from the forward's bf16 O
    own = (to_np(g["o"]) * to_np(inp["dO"])).sum(-1)
    assert np.allclose(to_np(g["delta"]), own, rtol=1e-5, atol=1e-5)


@pytest.mark.gpu
def test_atomic_backward_many_key_tiles_sampled():
    """B=1 H=4 N=2000 causal: dQ rows accumulate over up to 16 key tiles; sampled rows vs the oracle."""
    dev = cuda_or_skip()
    B, H, N, D = 1, 4, 2000, 128
    inp = make_qkv(B, H, N, D, seed=777, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    g = _run(inp, True, dev, scale, torch.float32)
    rows = sample_rows(B, H, N, 48, seed=777)
    ref_dq, _ = oracle.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["dO"], scale, True, rows)
    got = np.stack([to_np(g["dq"][b, h, i]) for b, h, i in rows])
    assert_close(got, ref_dq, TOL_BF16, what="sampled dq")


@pytest.mark.gpu
def test_atomic_backward_rejects_small_accumulator(lib):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    inp = make_qkv(1, 1, 256, 128, seed=3, dtype="bf16", with_dO=True)
    q, k, v, dO = (inp[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = fa.fa_forward(q, k, v)
    small = torch.empty(256 * 128 - 4, dtype=torch.float32, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_backward_atomic(q, k, v, o, dO, lse, dq_accum=small)
    assert e.value.code == nat.FA_ERR_WORKSPACE
