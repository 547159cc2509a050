"""The C ABI library builds, loads and exports every symbol include/lp.h declares;
host-side validation rejects bad arguments before any CUDA work (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lp():
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    import lm_head_linear_tcgen05_gb300 as mod
    mod.lib()
    return mod


def _declared():
    with open(os.path.join(ROOT, "include", "lp.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^LP_API\s+[^;]*?\b(lp_[a-z_]+)\s*\(", text, flags=re.M)))


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_header_declarations_match_binding_list(lp):
    assert _declared() == sorted(lp.EXPORTED)


def test_library_exports_every_declared_symbol(lp):
    L = lp.lib()
    for name in _declared():
        assert hasattr(L, name), name
    # and nothing but the C ABI has default visibility
    out = os.popen(f"nm -D --defined-only {lp.LIB_PATH}").read()
    exported = sorted(set(l.split()[-1] for l in out.splitlines() if " T " in l and "lp_" in l))
    assert exported == _declared()


def test_status_strings(lp):
    for code, name in lp.STATUS_NAMES.items():
        assert lp.lp_status_string(code).startswith(name)


def _part(lp, real, padded, bounds):
    return lp.VocabPartition(real, padded, tuple((bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)))


def test_workspace_sizes(lp):
    p = _part(lp, 1000, 1000, [0, 1000])
    # 4 vocabulary blocks of 256 ids x 64 rows x 4 bytes, three statistics, plus one target array
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, p) == 3 * 1024 + 256
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD_FROM_LOGITS, 64, 256, p) == 0
    assert lp.lp_workspace_size(lp.LP_OP_TOP_P_REPLAY, 64, 256, p) == 0
    assert lp.lp_workspace_size(lp.LP_OP_TOP_P_REPLAY_DENSE_MASK, 64, 256, p) == 64 * 64 * 4
    # padded ids need no vocabulary block: 152064 padded, 151936 real in 4 shards
    p4 = _part(lp, 151936, 152064, [0, 38016, 76032, 114048, 152064])
    nb = 149 + 149 + 149 + 148
    T = 4096
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, T, 4096, p4) == 3 * nb * T * 4 + T * 4
    # backward: G in bf16 [T, V] plus dX partials and db partials
    assert lp.lp_workspace_size(lp.LP_OP_BACKWARD, T, 4096, p4) > T * 151936 * 2
    # invalid partitions size to 0
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, _part(lp, 1000, 1000, [0, 500, 900])) == 0
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 0, 256, p) == 0


def _raw_forward(lp, X, T, H, W, part, y, tau, logp, lse, ws, wsb):
    L = lp.lib()
    cp, keep = lp._c_partition(part)
    Wa = (ctypes.c_void_p * max(len(W), 1))(*W)
    out = lp._Outputs(logp, lse, None, None)
    return L.lp_forward(X, T, H, Wa, None, ctypes.byref(cp), y, tau, ctypes.byref(out), ws, wsb, None)


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")
def test_host_validation_rejects_before_any_launch(lp):
    p = _part(lp, 1000, 1000, [0, 1000])
    A = 0x10000  # fake, 16-byte aligned; never dereferenced on the host
    ws = lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, p)
    ok_args = dict(X=A, T=64, H=256, W=[A], part=p, y=A, tau=0.7, logp=A, lse=A, ws=A, wsb=ws)

    def call(**kw):
        a = dict(ok_args)
        a.update(kw)
        return _raw_forward(lp, **a)

    assert call(X=None) == 1
    assert call(H=250) == 1                                  # H % 8 != 0
    assert call(T=-1) == 1
    assert call(T=0, X=None, y=None, W=[None], logp=None, lse=None, ws=None, wsb=0) == 0   # empty batch: no work
    assert call(T=0, tau=0.0) == 1                           # scalars are still checked
    assert call(tau=0.0) == 1
    assert call(tau=float("nan")) == 1
    assert call(tau=-1.0) == 1
    assert call(part=_part(lp, 1000, 1000, [0, 400, 900])) == 1   # does not cover [0, 1000)
    assert call(part=_part(lp, 1001, 1000, [0, 1000])) == 1       # vocab_real > vocab_padded
    assert call(part=_part(lp, 1000, 1000, [0, 600, 500, 1000])) == 1  # not ascending
    assert call(X=A + 8) == 2                                 # misaligned
    assert call(W=[A + 2]) == 2
    assert call(wsb=ws - 1) == 4
    # valid arguments reach the device check, which fails without a GPU
    assert call() == 3


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")
def test_replay_requires_null_entropy_and_nine_shards_rejected(lp):
    L = lp.lib()
    A = 0x10000
    p = _part(lp, 1000, 1000, [0, 1000])
    cp, keep = lp._c_partition(p)
    Wa = (ctypes.c_void_p * 1)(A)
    out = lp._Outputs(A, A, A, None)
    assert L.lp_top_p_replay(A, 4, 64, Wa, None, ctypes.byref(cp), A, A, 0.7, ctypes.byref(out), None, 0, None) == 1
    p9 = _part(lp, 900, 900, list(range(0, 901, 100)))
    cp9, keep9 = lp._c_partition(p9)
    out = lp._Outputs(A, A, None, None)
    Wa9 = (ctypes.c_void_p * 9)(*([A] * 9))
    assert L.lp_top_p_replay(A, 4, 64, Wa9, None, ctypes.byref(cp9), A, A, 0.7, ctypes.byref(out), None, 0,
                             None) == 1


def test_device_support_query_without_gpu(lp):
    if _has_gpu():
        pytest.skip("a GPU is present")
    assert lp.lp_device_supported() is False
