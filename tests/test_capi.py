"""The C ABI library builds, loads without a GPU, and exports every function
that include/moe.h declares (CPU only: no compute calls)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from ragged_grouped_gemm_topk_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = _declared()
    for want in ("moe_route_topk", "moe_permute", "moe_quantize_mxfp8_grouped", "moe_grouped_gemm_fwd",
                 "moe_grouped_gemm_dgrad", "moe_grouped_gemm_wgrad", "moe_unpermute_combine",
                 "moe_unpermute_combine_bwd", "moe_route_topk_bwd"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_declares_every_symbol():
    from ragged_grouped_gemm_topk_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == _declared()


def _declared_arity():
    """Parameter count of every moe_* function declared in include/*.h."""
    arity = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            src = re.sub(r"//[^\n]*", "", src)
            for name, params in re.findall(r"\b(moe_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
                params = params.strip()
                arity[name] = 0 if params in ("", "void") else len(params.split(","))
    return arity


def test_binding_prototypes_match_the_header():
    """The ctypes prototype of every entry point takes as many arguments as the
    header declares (a signature changed on one side only fails here, not at a call)."""
    from ragged_grouped_gemm_topk_gb300 import _lib
    arity = _declared_arity()
    assert sorted(arity) == _declared()
    wrong = {n: (len(_lib.SIGNATURES[n][1]), arity[n]) for n in arity if len(_lib.SIGNATURES[n][1]) != arity[n]}
    assert not wrong, wrong


def test_python_binding_has_every_entry_point_by_name():
    """One Python function per C entry point, same name (the error-string accessor
    is internal: failures surface as MoeError carrying its text)."""
    from ragged_grouped_gemm_topk_gb300 import binding
    missing = [n for n in _declared() if n != "moe_last_error_string" and not callable(getattr(binding, n, None))]
    assert not missing, missing


def test_host_only_calls(lib):
    lib.moe_version.restype = ctypes.c_int
    assert lib.moe_version() >= 0x100
    lib.moe_permute_workspace_size.restype = ctypes.c_size_t
    lib.moe_permute_workspace_size.argtypes = [ctypes.c_int] * 3
    assert lib.moe_permute_workspace_size(16384, 8, 256) == 64 * 256 * 4


def test_bad_arguments_rejected_before_any_launch():
    """Argument checks run on the host and return a status; nothing touches a GPU."""
    from ragged_grouped_gemm_topk_gb300 import _lib
    L = _lib.load()
    st = L.moe_route_topk(None, 10, 8, 9, 1, None, None, None, None, None)       # k > E
    assert st == _lib.MOE_ERR_INVALID_ARG
    assert b"k" in L.moe_last_error_string()
    a = _lib.Operand(None, _lib.MOE_BF16, None)
    b = _lib.Operand(None, _lib.MOE_F32, None)
    st = L.moe_grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(b), None, 16, 64, 48, 2, 0, None,
                                _lib.MOE_BF16, None, None, None)                  # K % 32
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = L.moe_quantize_mxfp8_grouped(None, _lib.MOE_BF16, 4, 48, None, 0, 0, None, None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = L.moe_quantize_mxfp8_grouped(None, _lib.MOE_BF16, 4, 64, None, 0, 1, None, None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG                                      # column-wise without groups
    st = L.moe_quantize_mxfp8_grouped(None, _lib.MOE_BF16, 4, 64, None, 0, 2, None, None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG                                      # tiled column-wise without groups
    st = L.moe_quantize_mxfp8_grouped(None, _lib.MOE_BF16, 4, 64, None, 0, 3, None, None, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED                                      # no such axis
    # gathered column-wise quantiser: row-wise axis, width, groups
    st = L.moe_quantize_mxfp8_gathered(None, _lib.MOE_BF16, 4, 64, 2, None, None, None, 2, 0, None, None, None,
                                       None)
    assert st == _lib.MOE_ERR_UNSUPPORTED                                      # axis 0 is not column-wise
    st = L.moe_quantize_mxfp8_gathered(None, _lib.MOE_BF16, 4, 48, 2, None, None, None, 2, 1, None, None, None,
                                       None)
    assert st == _lib.MOE_ERR_INVALID_ARG and b"K" in L.moe_last_error_string()   # K % 32
    st = L.moe_quantize_mxfp8_gathered(None, _lib.MOE_BF16, 4, 64, 2, None, None, None, 2, 2, None, None, None,
                                       None)
    assert st == _lib.MOE_ERR_INVALID_ARG                                      # K % 128 for tiled scales
    # combine backward with MXFP8 dYp: bf16 only, d % 32
    st = L.moe_unpermute_combine_bwd_mxfp8(None, None, _lib.MOE_BF16, 4, 40, 2, None, None, None, None, None,
                                           None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = L.moe_unpermute_combine_bwd_mxfp8(None, None, _lib.MOE_F32, 4, 64, 2, None, None, None, None, None,
                                           None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG


def test_no_cpu_fallback_in_product_package():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "ragged_grouped_gemm_topk_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
