"""Build liblp.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

    python -m lm_head_linear_tcgen05_gb300._build [--force] [-v] [--debug-bounds]

Objects go to lm_head_linear_tcgen05_gb300/_build/, the library to
lm_head_linear_tcgen05_gb300/liblp.so (both git-ignored). With --debug-bounds the same
sources are built with device-side bounds checks (LP_DEBUG_BOUNDS=1) into _build_debug/ and
liblp_debug.so, a stand-in for a sanitizer's out-of-bounds checks. The CUDA runtime is linked
statically and the driver API is reached through cudaGetDriverEntryPointByVersion,
so the library loads on a machine without a GPU driver (every call then returns
LP_ERR_UNSUPPORTED_DEVICE).

Provenance: the library embeds a hash of the sources and flags it was compiled from
(`lp_build_id()`), and a stamp file beside it records that hash and the machine it was
built on. A library is reused only when its stamp matches the current sources on this
machine; otherwise it is compiled again. `LAST_BUILD` says which happened, and the
binding refuses to load an in-tree library whose embedded hash differs from the sources.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import platform
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
CODE_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden"]
NVCC_FLAGS = CODE_FLAGS + ["-I" + INCLUDE, "-I" + CSRC]
DEBUG_FLAGS = ["-DLP_DEBUG_BOUNDS=1"]

# the most recent build() of this process: {"lib", "compiled", "source_hash", "machine"},
# and the latest such record of every library this process built or reused
LAST_BUILD: dict = {}
BUILDS: dict = {}


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


def source_hash(debug_bounds: bool = False) -> str:
    """Hash of every source and header (by path relative to the repository) and of the code
    flags: the identity of a build, the same on every machine."""
    srcs, headers = _inputs()
    h = hashlib.sha256()
    for f in srcs + headers:
        h.update(os.path.relpath(f, ROOT).replace(os.sep, "/").encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join(CODE_FLAGS + (DEBUG_FLAGS if debug_bounds else [])).encode())
    return h.hexdigest()[:16]


def _stamp_path(lib_path: str) -> str:
    return lib_path + ".stamp"


def _stamp(src_hash: str) -> dict:
    return {"source_hash": src_hash, "machine": platform.machine()}


def up_to_date(lib_path: str = LIB, debug_bounds: bool = False) -> bool:
    """True if lib_path exists and its stamp names the current sources and this machine."""
    if not os.path.exists(lib_path):
        return False
    try:
        with open(_stamp_path(lib_path)) as f:
            return json.load(f) == _stamp(source_hash(debug_bounds))
    except (OSError, ValueError):
        return False


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link liblp.so (liblp_debug.so with debug_bounds) unless an up-to-date build
    of the current sources for this machine exists; return its path. LAST_BUILD records
    whether it compiled."""
    lib_path, objdir = (DEBUG_LIB, DEBUG_OBJDIR) if debug_bounds else (LIB, OBJDIR)
    h = source_hash(debug_bounds)
    if not force and up_to_date(lib_path, debug_bounds):
        LAST_BUILD.clear()
        LAST_BUILD.update(lib=lib_path, compiled=False, **_stamp(h))
        BUILDS[lib_path] = dict(LAST_BUILD)
        return lib_path
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    srcs, _ = _inputs()
    extra = (DEBUG_FLAGS if debug_bounds else []) + [f'-DLP_SOURCE_HASH="{h}"']

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
    with open(_stamp_path(lib_path), "w") as f:
        json.dump(_stamp(h), f)
    LAST_BUILD.clear()
    LAST_BUILD.update(lib=lib_path, compiled=True, **_stamp(h))
    BUILDS[lib_path] = dict(LAST_BUILD)
    sys.stderr.write(f"{os.path.basename(lib_path)}: compiled from sources {h} on {platform.machine()}\n")
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true", help="build liblp_debug.so with device bounds checks")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug_bounds=a.debug_bounds))
    print(json.dumps(LAST_BUILD))
