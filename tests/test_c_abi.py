"""The boundary used from plain C: include/lp.h compiles as C99 and as C++17 on its own, a
C program (tests/c_abi_forward.c) builds and links against liblp.so and the CUDA runtime,
and on a GPU that program's lp_forward matches the fp64 oracle and the Python binding bit
for bit on the tiny configuration (T=64, H=256, V=1000, tau=1)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


@pytest.mark.parametrize("lang,std,comp", [("c", "-std=c99", "gcc"), ("c++", "-std=c++17", "g++")])
def test_header_compiles_standalone(tmp_path, lang, std, comp):
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "lp.h"\nint lp_header_probe(void) { return LP_MAX_SHARDS + (int)LP_OK; }\n')
    r = subprocess.run([_compiler(comp), std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", INCLUDE, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _build_c_program(tmp_path):
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    libdir = os.path.dirname(_build.LIB)
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("CUDA runtime headers not found")
    exe = tmp_path / "c_abi_forward"
    cmd = [_compiler("gcc"), "-std=c99", "-O2", "-Wall", "-Werror", "-I", INCLUDE, "-I",
           os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_abi_forward.c"), "-o", str(exe),
           "-L", libdir, "-llp", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_builds_and_links(tmp_path):
    exe = _build_c_program(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_program_forward_matches_oracle_and_binding(tmp_path):
    import torch

    import lm_head_linear_tcgen05_gb300 as lp
    import oracle
    from lp_util import TOL_ENT, TOL_LOGP, TOL_LSE, dev_inputs, max_abs, part_of
    exe = _build_c_program(tmp_path)
    T, H, V = 64, 256, 1000
    part = synth.even_partition(V, 1)
    inp = synth.forward_inputs(T, H, part, tau=1.0, seed=0)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(np.array([T, H, V], dtype="<i8").tobytes())
        f.write(np.array([inp.tau], dtype="<f4").tobytes())
        f.write(np.ascontiguousarray(inp.X, dtype="<u2").tobytes())
        f.write(np.ascontiguousarray(inp.W[0], dtype="<u2").tobytes())
        f.write(np.ascontiguousarray(inp.y, dtype="<i4").tobytes())
    r = subprocess.run([str(exe), str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(fout, dtype="<f4").reshape(3, T)
    ref = oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    assert max_abs(got[0], ref.logp) <= TOL_LOGP
    assert max_abs(got[1], ref.lse) <= TOL_LSE
    assert max_abs(got[2], ref.entropy) <= TOL_ENT
    # the same bits as the Python binding's call in this process
    torch.cuda.set_device(0)
    X, W, _, y = dev_inputs(inp)
    out = lp.lp_forward(X, W, None, part_of(part), y, inp.tau)
    for i, k in enumerate(("logp", "lse", "entropy")):
        assert np.array_equal(got[i], out[k].cpu().numpy()), k
