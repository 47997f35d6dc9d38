"""CPU-only checks of the C-ABI boundary: the library builds, loads and exports every entry
point include/fa.h declares (no compute call is made without a GPU)."""
import ctypes
import os
import re

from constrained_decoding_diffusion_gb300 import build, native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_calls():
    decl = declared_functions()
    assert set(native.EXPORTS) <= set(decl), decl
    assert set(decl) <= set(native.EXPORTS), decl


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    native.load(path)
    assert native.load() is not None


def test_last_error_without_gpu():
    lib = native.load()
    # a NULL handle is rejected on the host before any CUDA call
    rc = lib.fa_query(None, None, None, None, None, None, None)
    assert rc == native.FA_ERR_INVALID_ARG
    assert b"NULL" in lib.fa_last_error()
    n = ctypes.c_size_t()
    assert lib.fa_step_workspace_bytes(None, 1, 1, ctypes.byref(n)) == native.FA_ERR_INVALID_ARG


def test_oracle_and_product_share_no_sources():
    prod = set()
    for d, _, files in os.walk(os.path.join(ROOT, "constrained_decoding_diffusion_gb300", "csrc")):
        prod |= {f for f in files}
    orc = set(os.listdir(os.path.join(ROOT, "oracle")))
    assert not (prod & orc)
    for d, _, files in os.walk(os.path.join(ROOT, "constrained_decoding_diffusion_gb300")):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh")):
                src = open(os.path.join(d, f)).read()
                assert "import oracle" not in src and "from oracle" not in src and "oracle/" not in src, f
