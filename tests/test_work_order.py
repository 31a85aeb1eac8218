"""The causal work order by groups of heads, and the D = 64 forward's blocks drawn from a work counter.

A launch whose streamed operands exceed three quarters of L2 runs its causal tiles by groups of heads;
the D = 64 forward then draws its blocks from a per-launch counter that the launch zeroes again when it
ends.  These tests take a shape that is grouped (B=1 H=32 N=16384 D=64 causal: 128 MiB of K and V, more
than three quarters of the 129 MB L2) and
check that every tile is computed (outputs prefilled with NaN come back finite), that sampled rows match
the oracle, and that the counters leave nothing behind: repeated calls, calls on two streams at once,
and replays of a captured CUDA graph give bit-identical results.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BF16, TOL_LSE, BF16_REL, assert_close, cuda_or_skip
from synthetic_inputs import make_qkv, sample_rows

pytestmark = pytest.mark.gpu

SHAPE = (1, 32, 16384, 64)


def _inputs(dev, with_dO=False):
    B, H, N, D = SHAPE
    inp = make_qkv(B, H, N, D, seed=8080, dtype="bf16", with_dO=with_dO)
    return inp, {n: t.to(dev) for n, t in inp.items()}


def _nan_like(t, dtype=None):
    return torch.full_like(t, float("nan"), dtype=dtype or t.dtype)


def test_grouped_forward_covers_every_tile_and_matches_oracle():
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D = SHAPE
    inp, d = _inputs(dev)
    o = _nan_like(d["q"])
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    fa.fa_forward(d["q"], d["k"], d["v"], causal=True, o=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    scale = 1.0 / np.sqrt(D)
    rows = sample_rows(B, H, N, 96, seed=8080)
    ro, rl = oracle.forward_rows(inp["q"], inp["k"], inp["v"], scale, True, rows)
    idx = tuple(np.array(rows).T)
    assert_close(o[idx].double().cpu().numpy(), ro, TOL_BF16, BF16_REL, what="grouped O")
    assert_close(lse[idx].double().cpu().numpy(), rl, TOL_LSE, what="grouped LSE")


def test_grouped_forward_repeated_and_concurrent_calls_agree():
    """A counter left non-zero would make the next launch given it skip blocks (NaN rows here)."""
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    _, d = _inputs(dev)
    ref_o, ref_l = fa.fa_forward(d["q"], d["k"], d["v"], causal=True)
    for _ in range(3):
        o, l = fa.fa_forward(d["q"], d["k"], d["v"], causal=True)
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for s in (s1, s2):
        with torch.cuda.stream(s):
            outs.append(fa.fa_forward(d["q"], d["k"], d["v"], causal=True))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for o, l in outs:
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_grouped_backward_covers_every_tile_and_matches_oracle():
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D = SHAPE
    inp, d = _inputs(dev, with_dO=True)
    o, lse = fa.fa_forward(d["q"], d["k"], d["v"], causal=True)
    dq = _nan_like(d["q"], torch.float32)
    delta = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    dq, delta = fa.fa_backward_dq(d["q"], d["k"], d["v"], o, d["dO"], lse, causal=True, grad_dtype=torch.float32,
                                  dq=dq, delta=delta)
    dk, dv = _nan_like(d["k"], torch.float32), _nan_like(d["v"], torch.float32)
    fa.fa_backward_dkdv(d["q"], d["k"], d["v"], d["dO"], lse, delta, causal=True, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for name, t in (("dq", dq), ("delta", delta), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(t).all(), name
    scale = 1.0 / np.sqrt(D)
    rows = sample_rows(B, H, N, 48, seed=8081)
    rdq, _ = oracle.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["dO"], scale, True, rows)
    idx = tuple(np.array(rows).T)
    assert_close(dq[idx].double().cpu().numpy(), rdq, TOL_BF16, 0.0, what="grouped dQ")
    gen = torch.Generator().manual_seed(8082)
    krows = [(0, h, j) for h in (0, H - 1) for j in sorted({0, 127, 128, N - 1} |
                                                           {int(x) for x in torch.randint(0, N, (12,), generator=gen)})]
    rdk, rdv = oracle.backward_dkdv_rows(inp["q"], inp["k"], inp["v"], inp["dO"], scale, True, krows)
    kidx = tuple(np.array(krows).T)
    assert_close(dk[kidx].double().cpu().numpy(), rdk, TOL_BF16, 0.0, what="grouped dK")
    assert_close(dv[kidx].double().cpu().numpy(), rdv, TOL_BF16, 0.0, what="grouped dV")


def test_grouped_forward_in_a_cuda_graph_replays_identically():
    """A captured launch keeps its work counter; every replay must find it zeroed by the one before."""
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    _, d = _inputs(dev)
    ref_o, ref_l = fa.fa_forward(d["q"], d["k"], d["v"], causal=True)
    o, l = torch.empty_like(ref_o), torch.empty_like(ref_l)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fa_forward(d["q"], d["k"], d["v"], causal=True, o=o, lse=l)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_forward(d["q"], d["k"], d["v"], causal=True, o=o, lse=l)
    for _ in range(3):
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
