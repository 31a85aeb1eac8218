"""CPU checks of the C ABI: the library builds, loads, and exports every
function include/fa.h declares; the Python binding carries the same names.
No compute call is made (there may be no GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from helpers import ROOT

HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:FA_API\s+)?(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib_path():
    from attention_tiled_fwd_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("fa_forward", "fa_backward_dq", "fa_backward_dkdv", "fa_status_string", "fa_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared_functions():
        assert hasattr(lib, name), f"libfa.so does not export {name}"
    nm = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in nm.splitlines() if " T " in line}
    assert set(_declared_functions()) <= exported


def test_binding_lists_every_export(lib_path):
    from attention_tiled_fwd_gb300 import _native
    assert set(_declared_functions()) == set(_native.EXPORTS)
    import attention_tiled_fwd_gb300 as fa
    for n in ("fa_forward", "fa_backward_dq", "fa_backward_dkdv", "fa_device_status"):
        assert callable(getattr(fa, n))


def test_status_strings_need_no_gpu(lib_path):
    from attention_tiled_fwd_gb300 import _native
    lib = _native.load(lib_path)
    assert lib.fa_status_string(0) == b"ok"
    for code in range(-10, 0):
        s = lib.fa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.fa_version() >= 100


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "fa.h"\nint main(void){ return fa_version() > 0 ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c",
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_no_oracle_in_product_path():
    """The package never imports or links the oracle (the oracle is test infrastructure)."""
    pkg = os.path.join(ROOT, "attention_tiled_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fa_oracle" not in text, f


def test_product_fails_loudly_without_library(tmp_path):
    from attention_tiled_fwd_gb300 import _native
    with pytest.raises(ImportError):
        _native._lib_backup = _native._lib
        try:
            _native._lib = None
            _native.load(str(tmp_path / "missing.so"))
        finally:
            _native._lib = _native._lib_backup
