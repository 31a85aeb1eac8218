"""GPU split backward (dQ kernel, then dK/dV kernel) vs the float64 oracle,
through the C ABI.  The backward consumes the GPU forward's bf16 O and fp32
LSE, as a training step does; the oracle computes the exact gradient."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BF16, TOL_LSE, BF16_REL, assert_close, cuda_or_skip, to_np
from synthetic_inputs import WORKLOADS, make_qkv, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu


def _fwd_bwd(inp, causal, dev, scale, grad_dtype):
    import attention_tiled_fwd_gb300 as fa
    q, k, v, dO = (inp[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = fa.fa_forward(q, k, v, scale=scale, causal=causal)
    dq, delta = fa.fa_backward_dq(q, k, v, o, dO, lse, scale=scale, causal=causal, grad_dtype=grad_dtype)
    dk, dv = fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=scale, causal=causal, grad_dtype=grad_dtype)
    assert fa.fa_device_status() == 0
    return dict(o=o, lse=lse, dq=dq, delta=delta, dk=dk, dv=dv)


def _check_delta(g, inp, ref, rows=None):
    """D_i = rowsum(dO * O) is formed from the forward's bf16 O (as the pages' backward reads O).
    It must equal that row sum to fp32 accumulation accuracy, and differ from the oracle's D
    (built from the exact O) by no more than sum_d |dO_id| |O_id - O_exact,id|."""
    o = to_np(g["o"])
    do = to_np(inp["dO"])
    delta = to_np(g["delta"])
    own = (o * do).sum(-1)
    scale = (np.abs(o) * np.abs(do)).sum(-1)
    assert np.all(np.abs(delta - own) <= 1e-5 * scale + 1e-6), "delta is not rowsum(dO * O) of the GPU O"
    bound = (np.abs(do) * np.abs(o - ref["o"])).sum(-1) + 1e-5 * scale + 1e-6
    assert np.all(np.abs(delta - ref["delta"]) <= bound), "delta differs from the oracle beyond O's error"


SHAPES = [(1, 1, 1, 64), (1, 2, 77, 64), (1, 1, 128, 128), (2, 1, 300, 64), (1, 2, 257, 128),
          (1, 1, 520, 128), (1, 1, 640, 64)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_backward_small_shapes(shape, causal, grad_dtype):
    dev = cuda_or_skip()
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=200 + N + D, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    g = _fwd_bwd(inp, causal, dev, scale, grad_dtype)
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], scale, causal)
    rel = BF16_REL if grad_dtype == torch.bfloat16 else 0.0
    for n in ("dq", "dk", "dv"):
        assert_close(to_np(g[n]), ref[n], TOL_BF16, rel, what=f"{n} {shape} causal={causal}")
    _check_delta(g, inp, ref)
    assert_close(to_np(g["lse"]), ref["lse"], TOL_LSE, what="lse")


@pytest.mark.parametrize("shape", [(1, 2, 1100, 64), (1, 2, 900, 128)])
def test_backward_repeated_many_tiles(shape):
    """Many tiles per CTA in both backward kernels, several runs (pipeline-race check)."""
    dev = cuda_or_skip()
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=400 + N + D, dtype="bf16", with_dO=True)
    scale = 1.0 / np.sqrt(D)
    for causal in (False, True):
        ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["dO"], scale, causal)
        for rep in range(3):
            g = _fwd_bwd(inp, causal, dev, scale, torch.float32)
            for n in ("dq", "dk", "dv"):
                assert_close(to_np(g[n]), ref[n], TOL_BF16, what=f"{n} rep {rep} causal={causal}")


def test_backward_invariants_hold_on_gpu():
    """Column sums: sum_j dK_j = 0 (rows of dS sum to 0) and sum_j dV_j = sum_i dO_i."""
    dev = cuda_or_skip()
    inp = make_qkv(1, 2, 384, 64, seed=9, dtype="bf16", with_dO=True)
    g = _fwd_bwd(inp, True, dev, 0.125, torch.float32)
    dk = to_np(g["dk"]).sum(axis=2)
    dv = to_np(g["dv"]).sum(axis=2)
    assert np.abs(dk).max() < 0.05
    assert_close(dv, to_np(inp["dO"]).sum(axis=2), 0.05, what="sum dV")


def test_backward_is_deterministic():
    dev = cuda_or_skip()
    inp = make_qkv(1, 2, 700, 128, seed=4, dtype="bf16", with_dO=True)
    a = _fwd_bwd(inp, True, dev, 1 / np.sqrt(128), torch.float32)
    b = _fwd_bwd(inp, True, dev, 1 / np.sqrt(128), torch.float32)
    for n in ("dq", "dk", "dv", "delta"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("name,grad_dtype", [("bwd_bf16_b2h16n4096d128_causal", torch.float32),
                                             ("bwd_bf16_b2h16n4096d128_causal", torch.bfloat16),
                                             ("fwdbwd_bf16_b1h32n32768d64_causal", torch.bfloat16)])
def test_backward_full_size_sampled(name, grad_dtype):
    """Full-size backward in the benchmark's launch configuration: dQ on sampled query rows;
    dK / dV on sampled key rows of two heads (the oracle needs every row's LSE and D there)."""
    dev = cuda_or_skip()
    w = WORKLOADS[name]
    causal = w.causal[0]
    inp = workload_inputs(w)
    g = _fwd_bwd(inp, causal, dev, w.scale, grad_dtype)
    rel = BF16_REL if grad_dtype == torch.bfloat16 else 0.0
    rows = sample_rows(w.B, w.H, w.N, 128, seed=w.seed)
    rdq, rdelta = oracle.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["dO"], w.scale, causal, rows)
    idx = tuple(np.array(rows).T)
    assert_close(g["dq"][idx].double().cpu().numpy(), rdq, TOL_BF16, rel, what=f"{name} dQ")
    # D from the bf16 O: within sum_d |dO| |O_gpu - O_exact| of the oracle's D (see _check_delta)
    ro, _ = oracle.forward_rows(inp["q"], inp["k"], inp["v"], w.scale, causal, rows)
    o_rows = g["o"][idx].double().cpu().numpy()
    do_rows = inp["dO"][idx].double().numpy()
    d_gpu = g["delta"][idx].double().cpu().numpy()
    mag = (np.abs(o_rows) * np.abs(do_rows)).sum(-1)
    assert np.all(np.abs(d_gpu - (o_rows * do_rows).sum(-1)) <= 1e-5 * mag + 1e-6), f"{name} delta vs own O"
    bound = (np.abs(do_rows) * np.abs(o_rows - ro)).sum(-1) + 1e-5 * mag + 1e-6
    assert np.all(np.abs(d_gpu - rdelta) <= bound), f"{name} delta vs oracle"
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    gen = torch.Generator().manual_seed(w.seed + 5)
    krows = []
    for b, h in heads:
        js = {0, 1, 127, 128, w.N - 1} | {int(x) for x in torch.randint(0, w.N, (27,), generator=gen)}
        krows += [(b, h, j) for j in sorted(js)]
    rdk, rdv = oracle.backward_dkdv_rows(inp["q"], inp["k"], inp["v"], inp["dO"], w.scale, causal, krows)
    kidx = tuple(np.array(krows).T)
    assert_close(g["dk"][kidx].double().cpu().numpy(), rdk, TOL_BF16, rel, what=f"{name} dK")
    assert_close(g["dv"][kidx].double().cpu().numpy(), rdv, TOL_BF16, rel, what=f"{name} dV")
    for n in ("dq", "dk", "dv"):
        assert torch.isfinite(g[n]).all(), n
