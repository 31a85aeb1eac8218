"""ctypes view of libfa.so (the C ABI in include/fa.h).

Loading fails loudly if the library has not been built: there is no fallback
implementation of any entry point.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

# enum fa_dtype / fa_status (include/fa.h)
FA_F32, FA_BF16 = 0, 1
FA_OK = 0
FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEAD_DIM, FA_ERR_DTYPE, FA_ERR_ALIGN = -1, -2, -3, -4, -5
FA_ERR_SCALE, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_DEVICE_PTR, FA_ERR_DEVICE = -6, -7, -8, -9, -10
FA_ERR_WORKSPACE, FA_ERR_SCRATCH_LIMIT = -11, -12
FA_DECODE_NOALLOC_SCRATCH_BYTES = 16 << 20  # fa.h: fixed scratch of fa_decode_noalloc, per device

# Every symbol include/fa.h declares.
EXPORTS = ("fa_forward", "fa_backward_dq", "fa_backward_dkdv", "fa_backward_atomic", "fa_decode",
           "fa_decode_workspace_bytes",
           "fa_decode_noalloc", "fa_status_string", "fa_device_status", "fa_selftest_timeout", "fa_selftest_exp2", "fa_version")

_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libfa.so is not built ({path}); run `python -m attention_tiled_fwd_gb300.build` "
                          "or __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    lib.fa_forward.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _i, _p]
    lib.fa_backward_dq.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _i, _i, _p]
    lib.fa_backward_dkdv.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _i, _i, _p]
    lib.fa_backward_atomic.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, ctypes.c_size_t, _i, _i, _i, _i,
                                       _f, _i, _i, _i, _p]
    lib.fa_decode.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _f, _i, _p, ctypes.c_size_t, _p]
    lib.fa_decode_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_decode_noalloc.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _f, _i, _p]
    lib.fa_status_string.argtypes = [_i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_device_status.argtypes = [_p]
    lib.fa_selftest_timeout.argtypes = [_i, _p]
    lib.fa_selftest_exp2.argtypes = [_p, _p, _i, _p]
    lib.fa_version.argtypes = []
    for name in ("fa_forward", "fa_backward_dq", "fa_backward_dkdv", "fa_backward_atomic", "fa_decode", "fa_decode_workspace_bytes",
                 "fa_decode_noalloc", "fa_device_status",
                 "fa_selftest_timeout", "fa_selftest_exp2", "fa_version"):
        getattr(lib, name).restype = _i
    _lib = lib
    return lib


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().fa_status_string(code).decode()
        super().__init__(f"{where}: {msg} (status {code})")
        self.code = code


def check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FAError(code, where)
