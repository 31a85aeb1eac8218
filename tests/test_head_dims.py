"""Head dimensions beyond the 64 / 128 kernels, through the C ABI, against the
float64 oracle: every multiple of 8 up to 256 runs forward and backward.
D = 192 and 256 have kernels of their own width; any other D runs on the
next wider kernel (64, 128, 192 or 256) with the panel past D zero-filled by
the TMA, so these shapes also check that nothing is read or written past the
caller's D ("unlimited head dimension" of the metal-flash-attention page's
documentation section, here up to 256)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import BF16_REL, TOL_BF16, TOL_LSE, assert_close, assert_scaled, cuda_or_skip, to_np
from synthetic_inputs import WORKLOADS, make_qkv, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu


def _fwd_bwd(inp, causal, dev, scale, grad_dtype, guard=True):
    """Forward + split backward; with guard, outputs sit inside larger buffers filled with a sentinel so
    that a write past the row's D columns or past the tensor shows up."""
    import attention_tiled_fwd_gb300 as fa
    q, k, v, dO = (inp[n].to(dev) for n in ("q", "k", "v", "dO"))
    B, H, N, D = q.shape

    def guarded(dtype):
        if not guard:
            return torch.empty((B, H, N, D), dtype=dtype, device=dev), None
        buf = torch.full((B * H * N * D + 64,), 7.0, dtype=dtype, device=dev)
        return buf[:B * H * N * D].view(B, H, N, D), buf

    o, ob = guarded(torch.bfloat16)
    dq, qb = guarded(grad_dtype)
    dk, kb = guarded(grad_dtype)
    dv, vb = guarded(grad_dtype)
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal, o=o)
    dq, delta = fa.fa_backward_dq(q, k, v, o, dO, lse, scale=scale, causal=causal, dq=dq)
    dk, dv = fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=scale, causal=causal, dk=dk, dv=dv)
    assert fa.fa_device_status() == 0
    if guard:
        for name, b in (("o", ob), ("dq", qb), ("dk", kb), ("dv", vb)):
            tail = b[B * H * N * D:]
            assert bool((tail == 7.0).all()), f"{name}: written past the end of the tensor"
    return dict(o=o, lse=lse, dq=dq, delta=delta, dk=dk, dv=dv)


FWD_SHAPES = [(1, 1, 77, 8), (1, 2, 150, 16), (2, 1, 200, 32), (1, 1, 300, 40), (1, 2, 129, 72),
              (1, 1, 260, 96), (1, 1, 200, 104), (1, 1, 140, 136), (1, 2, 270, 160), (1, 1, 199, 200),
              (1, 1, 131, 248)]


@pytest.mark.parametrize("shape", FWD_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_forward_any_head_dim(shape, causal):
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=600 + N + D, dtype="bf16")
    scale = 1.0 / np.sqrt(D)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal)
    assert fa.fa_device_status() == 0
    ro, rl = oracle.forward(inp["q"], inp["k"], inp["v"], scale, causal)
    assert_close(to_np(o), ro, TOL_BF16, BF16_REL, what=f"O D={D}")
    assert_close(to_np(lse), rl, TOL_LSE, what=f"lse D={D}")


# D = 192 and 256 on their own kernels (several key and query tiles, ragged tails); other D padded
BWD_SHAPES = [(1, 1, 1, 192), (1, 2, 200, 192), (1, 1, 333, 192), (1, 1, 1, 256), (1, 2, 130, 256),
              (2, 1, 321, 256), (1, 1, 190, 32), (1, 2, 140, 40), (1, 1, 270, 96), (1, 1, 150, 160),
              (1, 1, 201, 200), (1, 1, 129, 248), (1, 1, 100, 8)]


@pytest.mark.parametrize("shape", BWD_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_backward_any_head_dim(shape, causal, grad_dtype):
    dev = cuda_or_skip()
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=700 + N + D, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    g = _fwd_bwd(inp, causal, dev, scale, grad_dtype)
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], scale, causal)
    rel = BF16_REL if grad_dtype == torch.bfloat16 else 0.0
    assert_close(to_np(g["o"]), ref["o"], TOL_BF16, BF16_REL, what=f"o D={D}")
    for n in ("dq", "dk", "dv"):
        assert_close(to_np(g[n]), ref[n], TOL_BF16, rel, what=f"{n} D={D} causal={causal}")
    own = (to_np(g["o"]) * to_np(inp["dO"])).sum(-1)
    mag = (np.abs(to_np(g["o"])) * np.abs(to_np(inp["dO"]))).sum(-1)
    assert np.all(np.abs(to_np(g["delta"]) - own) <= 1e-5 * mag + 1e-6), "delta is not rowsum(dO * O)"


def test_wide_head_backward_is_deterministic():
    dev = cuda_or_skip()
    inp = make_qkv(1, 2, 300, 256, seed=5, dtype="bf16", with_dO=True)
    a = _fwd_bwd(inp, True, dev, 1 / 16, torch.float32, guard=False)
    b = _fwd_bwd(inp, True, dev, 1 / 16, torch.float32, guard=False)
    for n in ("dq", "dk", "dv", "delta"):
        assert torch.equal(a[n], b[n]), n


def test_wide_head_backward_full_size_sampled():
    """B=1 H=8 N=8192 D=256 forward + backward in the benchmark's launch configuration: dQ on sampled
    query rows, dK / dV on sampled key rows of two heads, against the oracle."""
    dev = cuda_or_skip()
    w = WORKLOADS["fwdbwd_bf16_b1h8n8192d256"]
    causal = w.causal[0]
    inp = workload_inputs(w)
    g = _fwd_bwd(inp, causal, dev, w.scale, torch.bfloat16, guard=False)
    rows = sample_rows(w.B, w.H, w.N, 64, seed=w.seed)
    idx = tuple(np.array(rows).T)
    ro, rl = oracle.forward_rows(inp["q"], inp["k"], inp["v"], w.scale, causal, rows)
    assert_close(g["o"][idx].double().cpu().numpy(), ro, TOL_BF16, BF16_REL, what=f"{w.name} O")
    assert_close(g["lse"][idx].double().cpu().numpy(), rl, TOL_LSE, what=f"{w.name} LSE")
    rdq, _ = oracle.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["dO"], w.scale, causal, rows)
    assert_close(g["dq"][idx].double().cpu().numpy(), rdq, TOL_BF16, BF16_REL, what=f"{w.name} dQ")
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    gen = torch.Generator().manual_seed(w.seed + 5)
    krows = []
    for b, h in heads:
        js = {0, 1, 127, 128, w.N - 1} | {int(x) for x in torch.randint(0, w.N, (19,), generator=gen)}
        krows += [(b, h, j) for j in sorted(js)]
    rdk, rdv = oracle.backward_dkdv_rows(inp["q"], inp["k"], inp["v"], inp["dO"], w.scale, causal, krows)
    kidx = tuple(np.array(krows).T)
    assert_close(g["dk"][kidx].double().cpu().numpy(), rdk, TOL_BF16, BF16_REL, what=f"{w.name} dK")
    assert_close(g["dv"][kidx].double().cpu().numpy(), rdv, TOL_BF16, BF16_REL, what=f"{w.name} dV")
    # the std-0.5 inputs make O and every gradient ~0.02, below the flat bound itself: check each against
    # its own magnitude too (bf16 storage and fp32 accumulation stay well under 2 % of the largest value)
    for what, got, ref in (("O", g["o"][idx], ro), ("dQ", g["dq"][idx], rdq), ("dK", g["dk"][kidx], rdk),
                           ("dV", g["dv"][kidx], rdv)):
        assert_scaled(got.double().cpu().numpy(), ref, 0.02, what=f"{w.name} {what}")
