"""The MOE_DEBUG build (device-side invariant checks that write MOE_DEV_ASSERT into
the status word instead of trapping) builds in-tree beside the release library and
exports the same entry points (CPU only: no compute calls)."""

import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", h)).read(), flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_debug_build_exports_every_symbol():
    from ragged_grouped_gemm_topk_gb300 import build
    path = build.build(debug=True)
    assert path == build.LIB_DEBUG and path != build.LIB and os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(lib, name), name


def test_loader_picks_the_debug_build_from_the_environment(monkeypatch):
    from ragged_grouped_gemm_topk_gb300 import _lib, build
    monkeypatch.setenv("MOE_DEBUG", "1")
    assert _lib.lib_path() == build.LIB_DEBUG
    monkeypatch.setenv("MOE_DEBUG", "0")
    assert _lib.lib_path() == build.LIB
