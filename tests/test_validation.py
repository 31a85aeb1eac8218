"""Argument validation of the C ABI.  Shape, dtype, head-dimension, scale,
NULL and alignment checks run before any CUDA call, so these need no GPU;
the device-pointer and device-status checks run on the GPU."""
import ctypes
import math

import pytest

from attention_tiled_fwd_gb300 import _native as nat


@pytest.fixture(scope="module")
def lib():
    from attention_tiled_fwd_gb300 import build
    build.build()
    return nat.load()


A = 4096  # a fake, 16-byte-aligned address: validation must reject the call before touching it


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=8, D=64, scale=0.125, causal=0, dtype=nat.FA_BF16):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, None)


def test_forward_rejects_bad_shapes(lib):
    assert fwd(lib, B=0) == nat.FA_ERR_SHAPE
    assert fwd(lib, H=0) == nat.FA_ERR_SHAPE
    assert fwd(lib, N=0) == nat.FA_ERR_SHAPE
    assert fwd(lib, N=-5) == nat.FA_ERR_SHAPE
    assert fwd(lib, B=70000) == nat.FA_ERR_SHAPE
    assert fwd(lib, B=65535, H=65535, N=65535) == nat.FA_ERR_SHAPE


def test_forward_rejects_head_dims(lib):
    # bf16: any multiple of 8 up to 256
    for D in (0, 4, 12, 100, 252, 260, 264, 320, 512):
        assert fwd(lib, D=D) in (nat.FA_ERR_HEAD_DIM, nat.FA_ERR_SHAPE), D
    for D in (8, 16, 32, 96, 160, 200, 256):
        assert fwd(lib, D=D) not in (nat.FA_ERR_HEAD_DIM, nat.FA_ERR_SHAPE), D
    # fp32: any multiple of 4 up to 256
    for D in (2, 6, 50, 258, 260, 288):
        assert fwd(lib, D=D, dtype=nat.FA_F32) == nat.FA_ERR_HEAD_DIM, D


def test_forward_rejects_dtype_scale_null_align(lib):
    assert fwd(lib, dtype=7) == nat.FA_ERR_DTYPE
    assert fwd(lib, scale=math.inf) == nat.FA_ERR_SCALE
    assert fwd(lib, scale=math.nan) == nat.FA_ERR_SCALE
    assert fwd(lib, q=None) == nat.FA_ERR_NULL
    assert fwd(lib, lse=None) == nat.FA_ERR_NULL
    assert fwd(lib, o=A + 2) == nat.FA_ERR_ALIGN
    assert fwd(lib, k=A + 8) == nat.FA_ERR_ALIGN


def test_backward_rejects(lib):
    def dq(**kw):
        a = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, delta=A, dq=A, B=1, H=1, N=8, D=128, scale=0.1, causal=1,
                 dtype=nat.FA_BF16, grad=nat.FA_F32)
        a.update(kw)
        return lib.fa_backward_dq(a["q"], a["k"], a["v"], a["o"], a["dO"], a["lse"], a["delta"], a["dq"], a["B"],
                                  a["H"], a["N"], a["D"], a["scale"], a["causal"], a["dtype"], a["grad"], None)

    def dkdv(**kw):
        a = dict(q=A, k=A, v=A, dO=A, lse=A, delta=A, dk=A, dv=A, B=1, H=1, N=8, D=64, scale=0.1, causal=0,
                 dtype=nat.FA_BF16, grad=nat.FA_BF16)
        a.update(kw)
        return lib.fa_backward_dkdv(a["q"], a["k"], a["v"], a["dO"], a["lse"], a["delta"], a["dk"], a["dv"],
                                    a["B"], a["H"], a["N"], a["D"], a["scale"], a["causal"], a["dtype"],
                                    a["grad"], None)

    assert dq(D=264) == nat.FA_ERR_HEAD_DIM
    assert dq(D=36) == nat.FA_ERR_HEAD_DIM
    assert dq(D=256) != nat.FA_ERR_HEAD_DIM and dq(D=40) != nat.FA_ERR_HEAD_DIM
    assert dq(grad=5) == nat.FA_ERR_DTYPE
    assert dq(dtype=nat.FA_F32) == nat.FA_ERR_DTYPE
    assert dq(delta=None) == nat.FA_ERR_NULL
    assert dq(dO=A + 4) == nat.FA_ERR_ALIGN
    assert dq(N=0) == nat.FA_ERR_SHAPE
    assert dkdv(D=288) == nat.FA_ERR_HEAD_DIM
    assert dkdv(D=20) == nat.FA_ERR_HEAD_DIM
    assert dkdv(D=192) != nat.FA_ERR_HEAD_DIM
    assert dkdv(dv=None) == nat.FA_ERR_NULL
    assert dkdv(scale=float("inf")) == nat.FA_ERR_SCALE
    assert dkdv(lse=A + 12) == nat.FA_ERR_ALIGN


def test_selftest_rejects_bad_limit(lib):
    assert lib.fa_selftest_timeout(0, None) == nat.FA_ERR_SHAPE
    assert lib.fa_selftest_timeout(3_000_000, None) == nat.FA_ERR_SHAPE


# ----------------------------------------------------------------------------- GPU-side checks
@pytest.mark.gpu
def test_host_pointer_is_rejected_before_launch(lib):
    import torch
    from helpers import cuda_or_skip
    dev = cuda_or_skip()
    q = torch.randn(1, 1, 64, 64, device=dev).bfloat16()
    host = torch.empty(1, 1, 64, 64, dtype=torch.bfloat16)  # pageable host memory
    lse = torch.empty(1, 1, 64, device=dev)
    rc = lib.fa_forward(q.data_ptr(), q.data_ptr(), q.data_ptr(), host.data_ptr(), lse.data_ptr(), 1, 1, 64, 64,
                        0.125, 0, nat.FA_BF16, None)
    assert rc == nat.FA_ERR_DEVICE_PTR


@pytest.mark.gpu
def test_bounded_wait_times_out_and_reports(lib):
    """A wait on a barrier nothing arrives on ends after its limit and the status word says so;
    the context stays usable afterwards."""
    import torch
    from helpers import cuda_or_skip
    import attention_tiled_fwd_gb300 as fa
    dev = cuda_or_skip()
    assert fa.fa_device_status() == 0
    fa.fa_selftest_timeout(20000)  # 20 ms
    assert fa.fa_device_status() == nat.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == 0  # read clears it
    x = torch.ones(1024, device=dev)
    assert float(x.sum()) == 1024.0


@pytest.mark.gpu
def test_calls_from_a_fresh_thread():
    """Every entry point works from a thread that has made no CUDA call before (a worker thread,
    or autograd's backward thread)."""
    import threading
    import torch
    import attention_tiled_fwd_gb300 as fa
    from helpers import cuda_or_skip
    dev = cuda_or_skip()
    g = torch.Generator().manual_seed(5)
    q, k, v, dO = (torch.randn(1, 2, 200, 64, generator=g).bfloat16().to(dev) for _ in range(4))
    o_main, lse_main = fa.fa_forward(q, k, v, causal=True)
    out = {}

    def work():
        try:
            o, lse = fa.fa_forward(q, k, v, causal=True)
            dq, delta = fa.fa_backward_dq(q, k, v, o, dO, lse, causal=True, grad_dtype=torch.bfloat16)
            dk, dv = fa.fa_backward_dkdv(q, k, v, dO, lse, delta, causal=True, grad_dtype=torch.bfloat16)
            od, _ = fa.fa_decode(q[:, :, -1:].contiguous(), k, v, causal=True)
            torch.cuda.synchronize()
            out["r"] = (o, od)
        except Exception as e:  # reported in the main thread
            out["e"] = e

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert "e" not in out, out.get("e")
    o, od = out["r"]
    assert torch.equal(o, o_main)
    assert (od.float() - o_main[:, :, -1:].float()).abs().max().item() < 2e-2
