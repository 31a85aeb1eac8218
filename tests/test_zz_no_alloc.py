"""fa_decode_noalloc: decode with its partials in the library's fixed static
scratch instead of a caller workspace.  It runs the same kernels with the same
key split as fa_decode (the entry point with a caller workspace), so on
consecutive calls that reuse the scratch with different sizes and inputs its
results must equal fa_decode's bit for bit; both are also checked against the
float64 oracle's decode form, and the size limit is checked.  This file is
named to be collected last, so that the scratch has already been through the
other tests' process state when it runs in a full session; it also runs
alone."""
import ctypes
import os
import re

import pytest
import torch

import oracle
from attention_tiled_fwd_gb300 import _native as nat
from helpers import BF16_REL, ROOT, TOL_BF16, TOL_LSE, assert_close, cuda_or_skip


@pytest.fixture(scope="module")
def lib():
    from attention_tiled_fwd_gb300 import build
    build.build()
    return nat.load()


def test_scratch_limit_matches_header():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define\s+FA_DECODE_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == nat.FA_DECODE_NOALLOC_SCRATCH_BYTES


def test_oversize_is_rejected_before_launch(lib):
    # one chunk per (batch, head) once B*H is large, so the partials grow with B*H*n_q*(D+2)
    B, H, nq, N, D = 1, 4096, 16, 256, 128
    need = ctypes.c_size_t(0)
    assert lib.fa_decode_workspace_bytes(B, H, nq, N, D, ctypes.byref(need)) == nat.FA_OK
    assert need.value > nat.FA_DECODE_NOALLOC_SCRATCH_BYTES
    # the size check comes before the pointer checks and before any CUDA call
    rc = lib.fa_decode_noalloc(None, None, None, None, None, B, H, nq, N, D, 0.1, 1, None)
    assert rc == nat.FA_ERR_SCRATCH_LIMIT
    assert b"FA_DECODE_NOALLOC_SCRATCH_BYTES" in lib.fa_status_string(rc)
    # shape errors keep their own codes
    assert lib.fa_decode_noalloc(None, None, None, None, None, 1, 1, 17, 100, 128, 0.1, 0, None) == nat.FA_ERR_SHAPE
    assert lib.fa_decode_noalloc(None, None, None, None, None, 1, 1, 1, 100, 64, 0.1, 0, None) == nat.FA_ERR_NULL


def _case(B, H, nq, N, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, nq, D, generator=g).bfloat16().cuda()
    k = torch.randn(B, H, N, D, generator=g).bfloat16().cuda()
    v = torch.randn(B, H, N, D, generator=g).bfloat16().cuda()
    return q, k, v


def _call_noalloc(lib, q, k, v, causal):
    B, H, nq, D = q.shape
    N = k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, nq), float("nan"), dtype=torch.float32, device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, nq, N, D, D ** -0.5, int(causal), stream)
    assert rc == nat.FA_OK, lib.fa_status_string(rc)
    return o, lse


def _call_with_workspace(lib, q, k, v, causal):
    B, H, nq, D = q.shape
    N = k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, nq), float("nan"), dtype=torch.float32, device=q.device)
    need = ctypes.c_size_t(0)
    assert lib.fa_decode_workspace_bytes(B, H, nq, N, D, ctypes.byref(need)) == nat.FA_OK
    ws = torch.empty(max(need.value, 16), dtype=torch.uint8, device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, nq, N, D, D ** -0.5, int(causal), ws.data_ptr(), ws.numel(), stream)
    assert rc == nat.FA_OK, lib.fa_status_string(rc)
    return o, lse


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_consecutive_calls(lib):
    cuda_or_skip()
    # consecutive calls with different sizes and inputs: the second reuses the scratch the first
    # wrote, with another layout of chunks and rows
    cases = [((2, 8, 4, 3001, 128), True, 11), ((1, 16, 1, 5000, 64), False, 12),
             ((1, 4, 8, 777, 256), True, 13), ((2, 8, 4, 3001, 128), True, 14)]
    for (B, H, nq, N, D), causal, seed in cases:
        q, k, v = _case(B, H, nq, N, D, seed)
        o1, l1 = _call_noalloc(lib, q, k, v, causal)
        o2, l2 = _call_noalloc(lib, q, k, v, causal)
        ow, lw = _call_with_workspace(lib, q, k, v, causal)
        torch.cuda.synchronize()
        assert nat.load().fa_device_status(None) == nat.FA_OK
        _check_against_workspace_and_oracle(q, k, v, causal, [(o1, l1), (o2, l2)], (ow, lw))


def _check_against_workspace_and_oracle(q, k, v, causal, noalloc_results, workspace_result):
    ow, lw = workspace_result
    for o, l in noalloc_results:
        assert torch.isfinite(o.float()).all() and torch.isfinite(l).all()
        # same kernels, same split, same order of every sum: identical bits, so a stale or partial read
        # of the shared scratch cannot hide inside a tolerance
        assert torch.equal(o.view(torch.int16), ow.view(torch.int16)), "O differs from fa_decode's"
        assert torch.equal(l.view(torch.int32), lw.view(torch.int32)), "LSE differs from fa_decode's"
    D = q.shape[-1]
    ro, rl = oracle.forward_kv(q.cpu(), k.cpu(), v.cpu(), D ** -0.5, causal)
    assert_close(ow.float().cpu().numpy(), ro, TOL_BF16, BF16_REL, what="o vs oracle")
    assert_close(lw.cpu().numpy(), rl, TOL_LSE, what="lse vs oracle")


@pytest.mark.gpu
def test_noalloc_at_the_size_limit(lib):
    cuda_or_skip()
    # the largest n_q at D = 256 over many heads: partials close to (but within) the fixed scratch
    B, H, nq, N, D = 1, 1024, 8, 512, 256
    need = ctypes.c_size_t(0)
    assert lib.fa_decode_workspace_bytes(B, H, nq, N, D, ctypes.byref(need)) == nat.FA_OK
    assert nat.FA_DECODE_NOALLOC_SCRATCH_BYTES // 2 < need.value <= nat.FA_DECODE_NOALLOC_SCRATCH_BYTES
    q, k, v = _case(B, H, nq, N, D, 21)
    o1, l1 = _call_noalloc(lib, q, k, v, True)
    o2, l2 = _call_noalloc(lib, q, k, v, True)
    ow, lw = _call_with_workspace(lib, q, k, v, True)
    torch.cuda.synchronize()
    assert nat.load().fa_device_status(None) == nat.FA_OK
    _check_against_workspace_and_oracle(q, k, v, True, [(o1, l1), (o2, l2)], (ow, lw))
