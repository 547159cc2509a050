"""Build liblp.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

    python -m lm_head_linear_tcgen05_gb300._build [--force] [-v] [--debug-bounds]

Objects go to lm_head_linear_tcgen05_gb300/_build/, the library to
lm_head_linear_tcgen05_gb300/liblp.so (both git-ignored). With --debug-bounds the same
sources are built with device-side bounds checks (LP_DEBUG_BOUNDS=1) into _build_debug/ and
liblp_debug.so, a stand-in for a sanitizer's out-of-bounds checks. The CUDA runtime is linked
statically and the driver API is reached through cudaGetDriverEntryPointByVersion,
so the library loads on a machine without a GPU driver (every call then returns
LP_ERR_UNSUPPORTED_DEVICE).
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblp.so")
DEBUG_OBJDIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "liblp_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblp.so")
    return exe


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                     + glob.glob(os.path.join(INCLUDE, "*.h")))
    return srcs, headers


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    srcs, headers = _inputs()
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in srcs + headers + [__file__])


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link liblp.so (liblp_debug.so with debug_bounds) unless it is newer than
    every source; return its path."""
    lib_path, objdir = (DEBUG_LIB, DEBUG_OBJDIR) if debug_bounds else (LIB, OBJDIR)
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    srcs, _ = _inputs()
    extra = ["-DLP_DEBUG_BOUNDS=1"] if debug_bounds else []

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + extra + (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true", help="build liblp_debug.so with device bounds checks")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug_bounds=a.debug_bounds))
