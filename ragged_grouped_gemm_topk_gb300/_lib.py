"""ctypes loader for libmoe.so: declares the C ABI of include/moe.h.

The library must have been built (``ragged_grouped_gemm_topk_gb300.build.build()``);
there is no fallback of any kind when it is missing.
"""

from __future__ import annotations

import ctypes as C
import os

from . import build as _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = range(5)
MOE_F32, MOE_BF16, MOE_E4M3, MOE_E2M1 = 0, 1, 2, 3
MOE_EPI_NONE, MOE_EPI_SWIGLU, MOE_EPI_DSWIGLU = 0, 1, 2
MOE_DEV_NAN_LOGIT, MOE_DEV_BAD_INDEX, MOE_DEV_TIMEOUT, MOE_DEV_ASSERT = 1, 2, 4, 8

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_CUDA", 4: "MOE_ERR_WORKSPACE"}


class Operand(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("dtype", C.c_int), ("scales", C.c_void_p), ("tensor_scale", C.c_void_p)]


vp, i32, sz, st = C.c_void_p, C.c_int, C.c_size_t, C.c_int
OP = C.POINTER(Operand)

# name -> (restype, argtypes); one line per entry point of include/moe.h
SIGNATURES = {
    "moe_version": (C.c_int, []),
    "moe_last_error_string": (C.c_char_p, []),
    "moe_check_wait_timeout": (st, [vp, i32, vp]),
    "moe_debug_selftest": (st, [vp, C.POINTER(C.c_int), vp]),
    "moe_route_topk": (st, [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]),
    "moe_permute_workspace_size": (sz, [i32, i32, i32]),
    "moe_permute": (st, [vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, sz,
                         vp, vp]),
    "moe_permute_noalloc": (st, [vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp]),
    "moe_quantize_mxfp8_grouped": (st, [vp, i32, i32, i32, vp, i32, i32, vp, vp, vp]),
    "moe_grouped_gemm_fwd": (st, [OP, OP, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp]),
    "moe_grouped_gemm_fwd_mxfp8_out": (st, [OP, OP, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]),
    "moe_grouped_gemm_dgrad": (st, [OP, OP, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, vp]),
    "moe_quantize_mxfp8_transposed": (st, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "moe_quantize_mxfp8_gathered": (st, [vp, i32, i32, i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp]),
    "moe_route_topk_gemm": (st, [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
    "moe_quantize_nvfp4": (st, [vp, i32, i32, i32, vp, vp, vp, vp]),
    "moe_permute_nvfp4": (st, [vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
    "moe_grouped_gemm_dgrad_mxfp8": (st, [OP, OP, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]),
    "moe_grouped_gemm_wgrad": (st, [OP, OP, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp]),
    "moe_unpermute_combine": (st, [vp, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp]),
    "moe_permute_capacity_workspace_size": (sz, [i32, i32, i32]),
    "moe_permute_capacity": (st, [vp, i32, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
    "moe_unpermute_combine_capacity": (st, [vp, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp]),
    "moe_unpermute_combine_bwd": (st, [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
    "moe_unpermute_combine_bwd_mxfp8": (st, [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
    "moe_route_topk_bwd": (st, [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]),
}

_lib = None


def lib_path() -> str:
    """The library this process uses: the MOE_DEBUG build when the environment sets
    MOE_DEBUG=1 (device-side invariant checks into the status word), else the release one."""
    return _build.lib_for(debug=os.environ.get("MOE_DEBUG") == "1")


def load(path: str | None = None) -> C.CDLL:
    """Load libmoe.so (already built) and declare every entry point."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libmoe.so is not built ({p}); run ragged_grouped_gemm_topk_gb300.build.build()")
    lib = C.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def call(name: str, *args) -> None:
    lib = load()
    status = getattr(lib, name)(*args)
    if status != MOE_OK:
        raise MoeError(name, status, lib.moe_last_error_string().decode(errors="replace"))
