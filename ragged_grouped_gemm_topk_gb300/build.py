"""Build libmoe.so (all CUDA sources under csrc/) in-tree for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process, in parallel; the shared
library is linked into ``_build/``.  Rebuilds only when a source or header is
newer than the library.  ``debug=True`` (or MOE_DEBUG=1 in the environment) builds
the MOE_DEBUG variant instead, with its device-side invariant checks, into
``_build/debug/``.  Usage: ``python -m ragged_grouped_gemm_topk_gb300.build [--debug]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoe.so")
BUILD_DEBUG = os.path.join(BUILD, "debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libmoe.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h")))


def lib_for(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps() + [os.path.abspath(__file__)])


def _compile(src: str, extra, out_dir: str) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool | None = None) -> str:
    """Compile every csrc/*.cu for sm_103a and link _build/libmoe.so (the MOE_DEBUG
    variant into _build/debug/ when debug, which defaults to MOE_DEBUG=1 in the
    environment); return its path."""
    if debug is None:
        debug = os.environ.get("MOE_DEBUG") == "1"
    lib, out_dir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    flags = list(extra_flags) + (["-DMOE_DEBUG"] if debug else [])
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, out_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug=True if "--debug" in sys.argv else None)
