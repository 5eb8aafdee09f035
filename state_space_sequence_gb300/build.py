"""Build libdlr.so (all CUDA sources in csrc/) for sm_103a with nvcc, in-tree.

Each translation unit is compiled in parallel to an object file, then linked into
``state_space_sequence_gb300/_build/libdlr.so``. Rebuilds only when a source or header is newer
than the library. No CMake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libdlr.so")
# the bounds-checked build (DLR_BOUNDS_CHECK, relocatable device code): same sources, every
# guarded index checked on the device
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libdlr_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdlr.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    """Build libdlr.so, or with ``checked`` the bounds-checked libdlr_checked.so."""
    lib, bdir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checked:
        extra += ["-DDLR_BOUNDS_CHECK", "-rdc=true"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", *(["-rdc=true"] if checked else []), "-o", tmp, *objs,
           "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked="--checked" in sys.argv))
