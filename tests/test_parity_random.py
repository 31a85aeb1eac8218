"""Seeded random shapes for every kernel family against the float64 oracle:
batch, heads, sequence length (any N, not only tile multiples), causal flag,
head dimension and, for decode, the number of query rows.  The shapes are
drawn once from a fixed seed, so every run checks the same cases."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BF16, TOL_LSE, TOL_F32, BF16_REL, assert_close, cuda_or_skip, to_np
from synthetic_inputs import make_qkv

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(20261202)


def _draw(n, dims, n_max):
    out = []
    for _ in range(n):
        B = int(_rng.integers(1, 3))
        H = int(_rng.integers(1, 4))
        N = int(_rng.integers(1, n_max + 1))
        D = int(_rng.choice(dims))
        causal = bool(_rng.integers(0, 2))
        out.append((B, H, N, D, causal))
    return out


def _draw_each(n_per, dims, n_max):
    """n_per shapes for every head dimension in dims, the first of each causal and the second not."""
    out = []
    for D in dims:
        for i, (B, H, N, _, c) in enumerate(_draw(n_per, [D], n_max)):
            out.append((B, H, N, D, (i % 2 == 0) if i < 2 else c))
    return out


FWD_BF16 = _draw_each(3, [64, 128, 192, 256], 700)
FWD_F32 = _draw(4, [32, 64, 96, 128], 300)
BWD = _draw_each(4, [64, 128], 600)
ATOMIC = _draw(4, [128], 500)
DECODE = [(B, H, int(_rng.integers(1, 17)), N, int(_rng.choice([64, 128, 256])), c)
          for B, H, N, _, c in _draw(8, [64], 3000)]


@pytest.mark.parametrize("shape", FWD_BF16, ids=str)
def test_random_forward_bf16(shape):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D, causal = shape
    t = make_qkv(B, H, N, D, seed=N * 7 + D, dtype="bf16", std=0.5 if D == 256 else 1.0)
    scale = 1.0 / np.sqrt(D)
    o, lse = fa.fa_forward(*(t[n].to(dev) for n in ("q", "k", "v")), scale=scale, causal=causal)
    assert fa.fa_device_status() == 0
    ro, rl = oracle.forward(t["q"], t["k"], t["v"], scale, causal)
    assert_close(to_np(o), ro, TOL_BF16, BF16_REL, what=f"O {shape}")
    assert_close(to_np(lse), rl, TOL_LSE, what=f"LSE {shape}")


@pytest.mark.parametrize("shape", FWD_F32, ids=str)
def test_random_forward_f32(shape):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D, causal = shape
    t = make_qkv(B, H, N, D, seed=N * 11 + D, dtype="f32")
    scale = 1.0 / np.sqrt(D)
    o, lse = fa.fa_forward(*(t[n].to(dev) for n in ("q", "k", "v")), scale=scale, causal=causal)
    ro, rl = oracle.forward(t["q"], t["k"], t["v"], scale, causal)
    assert_close(to_np(o), ro, TOL_F32, what=f"O {shape}")
    assert_close(to_np(lse), rl, TOL_LSE, what=f"LSE {shape}")


@pytest.mark.parametrize("shape", BWD, ids=str)
def test_random_backward(shape):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D, causal = shape
    t = make_qkv(B, H, N, D, seed=N * 13 + D, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    q, k, v, dO = (t[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal)
    dq, delta = fa.fa_backward_dq(q, k, v, o, dO, lse, scale=scale, causal=causal, grad_dtype=torch.bfloat16)
    dk, dv = fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=scale, causal=causal, grad_dtype=torch.bfloat16)
    assert fa.fa_device_status() == 0
    ref = oracle.backward(t["q"], t["k"], t["v"], t["dO"], scale, causal)
    for n, g in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(to_np(g), ref[n], TOL_BF16, BF16_REL, what=f"{n} {shape}")


@pytest.mark.parametrize("shape", ATOMIC, ids=str)
def test_random_backward_atomic(shape):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D, causal = shape
    t = make_qkv(B, H, N, D, seed=N * 17 + D, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    q, k, v, dO = (t[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv, _ = fa.fa_backward_atomic(q, k, v, o, dO, lse, scale=scale, causal=causal,
                                          grad_dtype=torch.float32)
    assert fa.fa_device_status() == 0
    ref = oracle.backward(t["q"], t["k"], t["v"], t["dO"], scale, causal)
    for n, g in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(to_np(g), ref[n], TOL_BF16, what=f"{n} {shape}")


@pytest.mark.parametrize("shape", DECODE, ids=str)
def test_random_decode(shape):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, nq, N, D, causal = shape
    nq = min(nq, N)
    g = torch.Generator().manual_seed(N + nq)
    q = torch.randn(B, H, nq, D, generator=g).bfloat16()
    k = torch.randn(B, H, N, D, generator=g).bfloat16()
    v = torch.randn(B, H, N, D, generator=g).bfloat16()
    scale = 1.0 / np.sqrt(D)
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    assert fa.fa_device_status() == 0
    ro, rl = oracle.forward_kv(q, k, v, scale, causal)
    assert_close(to_np(o), ro, TOL_BF16, BF16_REL, what=f"decode O {shape}")
    assert_close(to_np(lse), rl, TOL_LSE, what=f"decode LSE {shape}")
