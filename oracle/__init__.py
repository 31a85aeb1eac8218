"""Float64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA path never
imports it and shares no code with it.

The arithmetic lives in ``fa_oracle.c`` (plain C, float64, one head per call,
full score rows, natural exp).  This module compiles it with gcc, loads it
with ctypes and loops over (batch, head) slices, optionally on several host
threads (ctypes releases the GIL during each foreign call; threading changes
which head runs where, never the arithmetic inside a head).

Conventions: arrays are ``[B, H, N, D]`` (or ``[B, H, N]`` for lse / delta),
C-contiguous float64 numpy arrays.  Inputs in another dtype are upcast
exactly (bf16 and f32 values are representable in float64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into a shared library (plain -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.fa_oracle_forward_rows.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_double, ctypes.c_int, ctypes.c_int64, _ip,
                                                   _dp, _dp]
            lib.fa_oracle_backward_head.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_double, ctypes.c_int, _dp, _dp, _dp,
                                                    _dp, _dp, _dp]
            lib.fa_oracle_backward_head_rows.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                                         ctypes.c_double, ctypes.c_int, ctypes.c_int64,
                                                         ctypes.c_int64, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.fa_oracle_backward_head_rows.restype = ctypes.c_int
            lib.fa_oracle_backward_dq_rows.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64,
                                                       ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                                       ctypes.c_int64, _ip, _dp, _dp]
            lib.fa_oracle_backward_dkdv_rows.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int64,
                                                         ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                                         ctypes.c_int64, _ip, _dp, _dp]
            lib.fa_oracle_forward_kv.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_double, ctypes.c_int, _dp, _dp]
            lib.fa_oracle_forward_kv.restype = ctypes.c_int
            for f in (lib.fa_oracle_forward_rows, lib.fa_oracle_backward_head,
                      lib.fa_oracle_backward_dq_rows, lib.fa_oracle_backward_dkdv_rows):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return a.ctypes.data_as(_dp) if a is not None else None


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed (rc={rc})")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _map_heads(fn, heads: Sequence[Tuple[int, int]], threads: Optional[int]):
    threads = default_threads() if threads is None else max(1, threads)
    if threads == 1 or len(heads) <= 1:
        for bh in heads:
            fn(bh)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fn, heads))


def forward(q, k, v, scale: float, causal: bool, threads: Optional[int] = None):
    """O [B,H,N,D] and natural LSE [B,H,N] of softmax(scale Q K^T) V, every row."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = q.shape
    o = np.empty((B, H, N, D))
    lse = np.empty((B, H, N))
    lib = _load()

    def one(bh):
        b, h = bh
        _check(lib.fa_oracle_forward_rows(_ptr(q[b, h]), _ptr(k[b, h]), _ptr(v[b, h]), N, D,
                                          float(scale), int(bool(causal)), N, None,
                                          _ptr(o[b, h]), _ptr(lse[b, h])), "forward")

    _map_heads(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return o, lse


def forward_kv(q, k, v, scale: float, causal: bool, threads: Optional[int] = None):
    """Decode form: q [B,H,n_q,D] against k, v [B,H,N_k,D]; the query rows are the last n_q
    positions (causal: row i sees keys j <= N_k - n_q + i).  Returns O [B,H,n_q,D], LSE [B,H,n_q]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, nq, D = q.shape
    nk = k.shape[2]
    o = np.empty((B, H, nq, D))
    lse = np.empty((B, H, nq))
    lib = _load()

    def one(bh):
        b, h = bh
        _check(lib.fa_oracle_forward_kv(_ptr(q[b, h]), _ptr(k[b, h]), _ptr(v[b, h]), nq, nk, D, float(scale),
                                        int(bool(causal)), _ptr(o[b, h]), _ptr(lse[b, h])), "forward_kv")

    _map_heads(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return o, lse


def backward(q, k, v, dO, scale: float, causal: bool, threads: Optional[int] = None):
    """Full plain-definition backward.  Returns dict o, lse, delta, dq, dk, dv (float64)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, N, D = q.shape
    out = {n: np.empty((B, H, N, D)) for n in ("o", "dq", "dk", "dv")}
    out["lse"] = np.empty((B, H, N))
    out["delta"] = np.empty((B, H, N))
    lib = _load()

    def one(bh):
        b, h = bh
        _check(lib.fa_oracle_backward_head(_ptr(q[b, h]), _ptr(k[b, h]), _ptr(v[b, h]),
                                           _ptr(dO[b, h]), N, D, float(scale), int(bool(causal)),
                                           _ptr(out["o"][b, h]), _ptr(out["lse"][b, h]),
                                           _ptr(out["delta"][b, h]), _ptr(out["dq"][b, h]),
                                           _ptr(out["dk"][b, h]), _ptr(out["dv"][b, h])), "backward")

    _map_heads(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return out


def backward_row_range(q, k, v, dO, scale: float, causal: bool, heads: Sequence[Tuple[int, int]],
                       row_begin: int, row_end: int, threads: Optional[int] = None):
    """Forward + backward terms of query rows [row_begin, row_end) for each listed (b, h) head.

    Returns {(b, h): dict(o, lse, delta, dq, dk, dv)} where o/lse/delta/dq hold those rows
    and dk/dv hold those rows' contributions (the full gradients when the range is 0..N).
    """
    D = q.shape[-1]
    N = q.shape[-2]
    lib = _load()
    out = {}

    def one(bh):
        b, h = bh
        qi, ki, vi, di = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(dO[b, h])
        r = {"o": np.zeros((N, D)), "lse": np.zeros((N,)), "delta": np.zeros((N,)),
             "dq": np.zeros((N, D)), "dk": np.zeros((N, D)), "dv": np.zeros((N, D))}
        _check(lib.fa_oracle_backward_head_rows(_ptr(qi), _ptr(ki), _ptr(vi), _ptr(di), N, D, float(scale),
                                                int(bool(causal)), int(row_begin), int(row_end),
                                                _ptr(r["o"]), _ptr(r["lse"]), _ptr(r["delta"]), _ptr(r["dq"]),
                                                _ptr(r["dk"]), _ptr(r["dv"])), "backward_row_range")
        for n in ("o", "lse", "delta", "dq"):
            r[n] = r[n][row_begin:row_end]
        out[bh] = r

    _map_heads(one, list(heads), threads)
    return out


def _group_rows(rows: Iterable[Tuple[int, int, int]]):
    groups = {}
    for idx, (b, h, i) in enumerate(rows):
        groups.setdefault((int(b), int(h)), []).append((idx, int(i)))
    return groups


def forward_rows(q, k, v, scale: float, causal: bool, rows: Sequence[Tuple[int, int, int]],
                 threads: Optional[int] = None):
    """O and LSE for selected (b, h, i) query rows: arrays [len(rows), D] and [len(rows)].

    ``q, k, v`` may be torch tensors of the run dtype; only the heads named in
    ``rows`` are upcast.
    """
    rows = list(rows)
    D = q.shape[-1]
    N = q.shape[-2]
    o = np.empty((len(rows), D))
    lse = np.empty((len(rows),))
    lib = _load()
    groups = _group_rows(rows)

    def one(bh):
        b, h = bh
        idx = groups[bh]
        qi, ki, vi = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h])
        ids = np.array([i for _, i in idx], dtype=np.int64)
        oo = np.empty((len(ids), D))
        ll = np.empty((len(ids),))
        _check(lib.fa_oracle_forward_rows(_ptr(qi), _ptr(ki), _ptr(vi), N, D, float(scale),
                                          int(bool(causal)), len(ids), ids.ctypes.data_as(_ip),
                                          _ptr(oo), _ptr(ll)), "forward_rows")
        for n, (pos, _) in enumerate(idx):
            o[pos] = oo[n]
            lse[pos] = ll[n]

    _map_heads(one, list(groups.keys()), threads)
    return o, lse


def backward_dq_rows(q, k, v, dO, scale: float, causal: bool, rows: Sequence[Tuple[int, int, int]],
                     threads: Optional[int] = None):
    """dQ [len(rows), D] and D_i [len(rows)] for selected (b, h, i) query rows."""
    rows = list(rows)
    D = q.shape[-1]
    N = q.shape[-2]
    dq = np.empty((len(rows), D))
    delta = np.empty((len(rows),))
    lib = _load()
    groups = _group_rows(rows)

    def one(bh):
        b, h = bh
        idx = groups[bh]
        qi, ki, vi, di = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(dO[b, h])
        ids = np.array([i for _, i in idx], dtype=np.int64)
        gq = np.empty((len(ids), D))
        dd = np.empty((len(ids),))
        _check(lib.fa_oracle_backward_dq_rows(_ptr(qi), _ptr(ki), _ptr(vi), _ptr(di), N, D,
                                              float(scale), int(bool(causal)), len(ids),
                                              ids.ctypes.data_as(_ip), _ptr(gq), _ptr(dd)),
               "backward_dq_rows")
        for n, (pos, _) in enumerate(idx):
            dq[pos] = gq[n]
            delta[pos] = dd[n]

    _map_heads(one, list(groups.keys()), threads)
    return dq, delta


def backward_dkdv_rows(q, k, v, dO, scale: float, causal: bool, rows: Sequence[Tuple[int, int, int]],
                       threads: Optional[int] = None):
    """dK, dV [len(rows), D] for selected (b, h, j) key rows.

    For every head named in ``rows`` this first computes the natural LSE and
    D_i of all N query rows with this oracle (forward_rows / dq_rows over the
    whole head), so it costs about 3 N^2 D multiply-adds per head.
    """
    rows = list(rows)
    D = q.shape[-1]
    N = q.shape[-2]
    dk = np.empty((len(rows), D))
    dv = np.empty((len(rows), D))
    lib = _load()
    groups = _group_rows(rows)
    heads = list(groups.keys())
    threads = default_threads() if threads is None else threads
    # per head: LSE and D of all query rows, split over row chunks for parallelism
    stats = {}
    for bh in heads:
        b, h = bh
        qi, ki, vi, di = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(dO[b, h])
        lse = np.empty((N,))
        delta = np.empty((N,))
        ochunk = np.empty((N, D))
        dqs = np.empty((N, D))
        nchunk = max(1, min(threads * 4, N))
        bounds = np.linspace(0, N, nchunk + 1).astype(np.int64)

        def chunk(c, qi=qi, ki=ki, vi=vi, di=di, lse=lse, delta=delta, ochunk=ochunk, dqs=dqs):
            lo, hi = int(bounds[c]), int(bounds[c + 1])
            if hi <= lo:
                return
            ids = np.arange(lo, hi, dtype=np.int64)
            _check(lib.fa_oracle_forward_rows(_ptr(qi), _ptr(ki), _ptr(vi), N, D, float(scale),
                                              int(bool(causal)), hi - lo, ids.ctypes.data_as(_ip),
                                              _ptr(ochunk[lo:hi]), _ptr(lse[lo:hi])), "forward_rows")
            _check(lib.fa_oracle_backward_dq_rows(_ptr(qi), _ptr(ki), _ptr(vi), _ptr(di), N, D,
                                                  float(scale), int(bool(causal)), hi - lo,
                                                  ids.ctypes.data_as(_ip), _ptr(dqs[lo:hi]),
                                                  _ptr(delta[lo:hi])), "backward_dq_rows")

        _map_heads(chunk, list(range(nchunk)), threads)
        stats[bh] = (qi, ki, vi, di, lse, delta)

    def one(bh):
        idx = groups[bh]
        qi, ki, vi, di, lse, delta = stats[bh]
        ids = np.array([j for _, j in idx], dtype=np.int64)
        gk = np.empty((len(ids), D))
        gv = np.empty((len(ids), D))
        _check(lib.fa_oracle_backward_dkdv_rows(_ptr(qi), _ptr(ki), _ptr(vi), _ptr(di), _ptr(lse),
                                                _ptr(delta), N, D, float(scale), int(bool(causal)),
                                                len(ids), ids.ctypes.data_as(_ip), _ptr(gk), _ptr(gv)),
               "backward_dkdv_rows")
        for n, (pos, _) in enumerate(idx):
            dk[pos] = gk[n]
            dv[pos] = gv[n]

    _map_heads(one, heads, threads)
    return dk, dv
