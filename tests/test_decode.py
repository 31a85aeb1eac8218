"""Decode (a few query rows against a long key/value range) vs the float64
oracle's decode form, through the C ABI.  The query rows are the last n_q
positions; causal row i sees keys j <= N - n_q + i."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_tiled_fwd_gb300 import _native as nat
from helpers import TOL_BF16, TOL_LSE, BF16_REL, assert_close, cuda_or_skip, to_np


def _inputs(B, H, nq, N, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, nq, D, generator=g).bfloat16()
    k = torch.randn(B, H, N, D, generator=g).bfloat16()
    v = torch.randn(B, H, N, D, generator=g).bfloat16()
    return q, k, v


# ------------------------------------------------------------------ host-side checks (no GPU)
@pytest.fixture(scope="module")
def lib():
    from attention_tiled_fwd_gb300 import build
    build.build()
    return nat.load()


def test_workspace_size_query(lib):
    out = ctypes.c_size_t(0)
    assert lib.fa_decode_workspace_bytes(2, 3, 4, 5000, 128, ctypes.byref(out)) == nat.FA_OK
    # O, m, l partials: 4 bytes x B x H x chunks x n_q x (D + 2), at least one chunk
    assert out.value >= 4 * 2 * 3 * 4 * 130 and out.value % (4 * 2 * 3 * 4 * 130) == 0
    assert lib.fa_decode_workspace_bytes(1, 1, 17, 100, 128, ctypes.byref(out)) == nat.FA_ERR_SHAPE
    assert lib.fa_decode_workspace_bytes(1, 1, 17, 100, 256, ctypes.byref(out)) == nat.FA_ERR_SHAPE
    assert lib.fa_decode_workspace_bytes(1, 1, 5, 4, 64, ctypes.byref(out)) == nat.FA_ERR_SHAPE  # n_q > N
    assert lib.fa_decode_workspace_bytes(1, 1, 1, 100, 96, ctypes.byref(out)) == nat.FA_ERR_HEAD_DIM
    assert lib.fa_decode_workspace_bytes(1, 1, 1, 100, 64, None) == nat.FA_ERR_NULL


def test_decode_rejects_before_launch(lib):
    A = 4096
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, nq=1, N=64, D=128, scale=0.1, causal=0, ws=A, wsb=1 << 20)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return lib.fa_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["nq"], a["N"], a["D"],
                             a["scale"], a["causal"], a["ws"], a["wsb"], None)

    assert call(nq=0) == nat.FA_ERR_SHAPE
    assert call(nq=17) == nat.FA_ERR_SHAPE
    assert call(D=32) == nat.FA_ERR_HEAD_DIM
    assert call(scale=float("nan")) == nat.FA_ERR_SCALE
    assert call(ws=None) == nat.FA_ERR_NULL
    assert call(k=A + 8) == nat.FA_ERR_ALIGN


# ------------------------------------------------------------------ GPU parity
# every (n_q <= 4, D) pair, n_q 5..16 in blocks of 4 rows (ragged last block), ragged chunk ends,
# n_q = N, and one long single-head cache that is cut into many chunks
SHAPES = [(1, 1, 1, 1, 64), (2, 3, 1, 1000, 128), (1, 3, 1, 5000, 256), (1, 2, 2, 70000, 64),
          (2, 1, 2, 3333, 128), (1, 1, 2, 300, 256), (1, 2, 3, 999, 64), (1, 1, 3, 2500, 128),
          (1, 1, 3, 129, 256), (1, 1, 4, 1500, 64), (1, 2, 4, 4133, 128), (2, 1, 4, 640, 256),
          (1, 1, 4, 4, 128), (1, 1, 16, 777, 64), (1, 2, 8, 2000, 256), (2, 2, 16, 16, 128),
          (1, 1, 5, 300, 128), (1, 1, 13, 1000, 256), (1, 2, 9, 8191, 128), (1, 1, 1, 200003, 128)]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_decode_matches_oracle(shape, causal):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, nq, N, D = shape
    q, k, v = _inputs(B, H, nq, N, D, seed=500 + N + D + nq)
    scale = 1.0 / np.sqrt(D)
    need = fa.fa_decode_workspace_bytes(B, H, nq, N, D)
    ws = torch.full((need // 4 + 4,), float("nan"), device=dev)  # garbage: the kernels must not need clearing
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal, workspace=ws)
    assert fa.fa_device_status() == 0
    ro, rl = oracle.forward_kv(q, k, v, scale, causal)
    assert_close(to_np(o), ro, TOL_BF16, BF16_REL, what=f"decode O {shape} causal={causal}")
    assert_close(to_np(lse), rl, TOL_LSE, what=f"decode LSE {shape} causal={causal}")


@pytest.mark.gpu
def test_decode_long_kv_cache_and_determinism():
    """A 32K-entry cache over 4 x 16 heads, single query row: checked in full, twice bit-identical."""
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, nq, N, D = 4, 16, 1, 32768, 128
    q, k, v = _inputs(B, H, nq, N, D, seed=77)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.fa_decode(qd, kd, vd, causal=True)
    o2, l2 = fa.fa_decode(qd, kd, vd, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = oracle.forward_kv(q, k, v, 1.0 / np.sqrt(D), True)
    assert_close(to_np(o1), ro, TOL_BF16, BF16_REL, what="decode 32K O")
    assert_close(to_np(l1), rl, TOL_LSE, what="decode 32K LSE")


@pytest.mark.gpu
def test_decode_rejects_small_workspace():
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    q, k, v = (t.to(dev) for t in _inputs(1, 2, 1, 3000, 128, seed=1))
    need = fa.fa_decode_workspace_bytes(1, 2, 1, 3000, 128)
    small = torch.empty(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_decode(q, k, v, workspace=small)
    assert e.value.code == nat.FA_ERR_WORKSPACE
