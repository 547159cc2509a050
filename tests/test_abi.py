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


def test_build_provenance(lp):
    # the loaded library carries the hash of the sources beside it; a second build() of
    # unchanged sources reuses it and says so
    from lm_head_linear_tcgen05_gb300 import _build
    assert lp.lp_build_id() == _build.source_hash()
    _build.build()
    assert _build.LAST_BUILD["compiled"] is False
    assert _build.LAST_BUILD["source_hash"] == lp.lp_build_id()
    info = lp.build_info()
    assert info["build_id"] == _build.source_hash() and info["compiled_in_this_process"] is False
    # the bounds-checked build hashes differently (its flags differ)
    assert _build.source_hash(debug_bounds=True) != _build.source_hash()


def test_wait_limit_range(lp):
    L = lp.lib()
    assert L.lp_set_wait_limit(999) == 1 and L.lp_set_wait_limit(10_000_000_001) == 1
    assert L.lp_set_wait_limit(1000) == 0 and L.lp_set_wait_limit(10_000_000_000) == 0
    assert L.lp_set_wait_limit(0) == 0                   # the 2 s default again


def test_status_strings(lp):
    for code, name in lp.STATUS_NAMES.items():
        assert lp.lp_status_string(code).startswith(name)


def test_bounds_checked_build_builds_and_says_so(lp):
    # the regular library reports no checks; the bounds-checked one (built from the same
    # sources with LP_DEBUG_BOUNDS=1) exports the same C ABI and reports them
    from lm_head_linear_tcgen05_gb300 import _build
    path = _build.build(debug_bounds=True)
    assert lp.lib().lp_debug_bounds_build() == 0
    D = ctypes.CDLL(path)
    assert D.lp_debug_bounds_build() == 1
    for name in _declared():
        assert hasattr(D, name), name
    if not _has_gpu():
        assert D.lp_selftest_bounds(None) == 3     # LP_ERR_UNSUPPORTED_DEVICE without a GPU


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


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")
def test_logits_backward_host_validation(lp):
    L = lp.lib()
    A, B = 0x100000, 0x900000          # fake, 16-byte aligned, far apart; never dereferenced on the host
    p = _part(lp, 90, 96, [0, 48, 96])
    cp, keep = lp._c_partition(p)
    T = 4
    assert lp.lp_workspace_size(lp.LP_OP_BACKWARD_FROM_LOGITS, T, 0, p) == 0

    def call(logits=(A, A + 4096), ld=(48, 48), out=(B, B + 4096), ld_out=(48, 48), dtype=lp.LP_DTYPE_BF16,
             ent=None, gent=None, T=T, tau=0.7):
        Lg = (ctypes.c_void_p * 2)(*logits)
        O = (ctypes.c_void_p * 2)(*out)
        ldv = (ctypes.c_int64 * 2)(*ld)
        ldo = (ctypes.c_int64 * 2)(*ld_out)
        return L.lp_backward_from_logits(Lg, ldv, T, ctypes.byref(cp), A, tau, A, A, ent, gent, O, ldo, dtype, None)

    assert call(dtype=2) == 1                                   # unknown output type
    assert call(ent=A) == 1                                     # entropy without its gradient
    assert call(ld=(40, 48)) == 1                               # row stride below the shard width
    assert call(ld=(52, 48)) == 2                               # row stride not a multiple of 8
    assert call(out=(B + 8, B + 4096)) == 2                     # misaligned output
    assert call(ld_out=(52, 48)) == 2                           # bf16 rows need a stride % 8 == 0 ...
    assert call(dtype=lp.LP_DTYPE_F32, ld_out=(52, 48)) == 3    # ... fp32 rows a stride % 4 == 0
    assert call(out=(A + 4096, B)) == 1                         # shard 0's output over shard 1's logits
    assert call(out=(B, B + 16)) == 1                           # outputs overlapping each other
    assert call(out=(A, A + 4096), dtype=lp.LP_DTYPE_F32) == 1  # fp32 over bf16 logits is not in place
    assert call(out=(A, A + 4096), ld_out=(56, 48)) == 1        # in place needs the same row stride
    assert call(out=(A, A + 4096)) == 3                         # in place: valid, reaches the device check
    assert call(T=0, logits=(None, None), out=(None, None)) == 0   # empty batch: no work
    assert call(T=0, tau=0.0) == 1
    assert call() == 3                                          # valid: fails only for want of a GPU


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")
def test_backward_ex_host_validation(lp):
    L = lp.lib()
    A = 0x100000
    p = _part(lp, 1000, 1000, [0, 1000])
    cp, keep = lp._c_partition(p)
    ws = lp.lp_workspace_size(lp.LP_OP_BACKWARD, 64, 256, p)

    def call(dx_dtype=0, accumulate=0, T=64, opts=True, dw_dtype=0):
        Wa = (ctypes.c_void_p * 1)(A)
        dW = (ctypes.c_void_p * 1)(A)
        o = lp._BackwardOptions(dx_dtype, accumulate, dw_dtype)
        return L.lp_backward_ex(A, T, 256, Wa, None, ctypes.byref(cp), A, 0.7, A, A, None, None, A, dW, None,
                                ctypes.byref(o) if opts else None, A, ws, None)

    assert call(dx_dtype=2) == 1
    assert call(dx_dtype=-1) == 1
    assert call(accumulate=2) == 1
    assert call(dw_dtype=3) == 1
    assert call(accumulate=1, dw_dtype=1) == 1  # accumulation needs fp32 dW
    assert call(dw_dtype=1, dx_dtype=1) == 3
    assert call(T=0, accumulate=1) == 0       # empty batch, accumulating: nothing to add, no device needed
    assert call(T=0) == 3                     # empty batch, overwriting: zeroes dW on the device
    assert call(dx_dtype=1, accumulate=1) == 3
    assert call(opts=False) == 3


@pytest.mark.skipif(_has_gpu(), reason="uses fake pointers; only safe without a GPU")
def test_forward_host_validation(lp):
    L = lp.lib()
    A = 0x100000  # fake device / host addresses; never dereferenced before the checks fail
    p = _part(lp, 1000, 1000, [0, 1000])
    cp, keep = lp._c_partition(p)
    T, H = 64, 256
    need = lp.lp_workspace_size(lp.LP_OP_FORWARD_HOST, T, H, p)
    # forward workspace + X + y + logp/lse/entropy + shard statistics, each 256-byte aligned
    assert need == lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, p) + T * H * 2 + 4 * 256 + 768
    Wa = (ctypes.c_void_p * 1)(A)

    def call(X=A, y=A, logp=A, lse=A, ws=A, wsb=need, T=T):
        out = lp._Outputs(logp, lse, None, None)
        return L.lp_forward_host(X, T, H, Wa, None, ctypes.byref(cp), y, 0.7, ctypes.byref(out), ws, wsb, None)

    assert call(X=None) == 1
    assert call(y=None) == 1
    assert call(lse=None) == 1
    assert call(wsb=need - 1) == 4
    assert call(ws=A + 8) == 2
    assert call(T=0, X=None, y=None, logp=None, lse=None, ws=None, wsb=0) == 0
    assert call() == 3                       # valid: fails only for want of a GPU, before any copy


def _local(lp, real, padded, bounds):
    return lp.VocabPartition(real, padded, tuple((bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)),
                             local=True)


def test_rank_local_partitions_validate(lp):
    # a rank-local partition tiles one rank's range [lo, hi) inside [0, vocab_padded)
    ok = _local(lp, 151936, 152064, [38016, 76032])
    nb = 149
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, ok) == 3 * nb * 64 * 4 + 256
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, _local(lp, 151936, 152064, [114048, 152064])) > 0
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, _local(lp, 151936, 152064, [0, 152064])) > 0
    # beyond the padded vocabulary, a negative start, a gap: rejected (size 0)
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, _local(lp, 151936, 152064, [114048, 152065])) == 0
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, _local(lp, 1000, 1000, [-8, 500])) == 0
    bad = lp.VocabPartition(1000, 1000, ((0, 400), (500, 1000)), local=True)
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, bad) == 0
    # the same ranges without the flag do not cover the vocabulary
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, 64, 256,
                                lp.VocabPartition(151936, 152064, ((38016, 76032),))) == 0
    # a flag other than 0 / 1 is rejected
    cp, keep = lp._c_partition(ok)
    cp.local = 2
    assert lp.lib().lp_workspace_size(lp.LP_OP_FORWARD, 64, 256, ctypes.byref(cp)) == 0


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")
def test_merge_and_sum_host_validation(lp):
    L = lp.lib()
    A, B = 0x100000, 0x900000            # fake, 16-byte aligned, far apart; never dereferenced on the host
    p = _part(lp, 1000, 1000, [0, 400, 1000])
    cp, keep = lp._c_partition(p)

    def merge(stats=A, T=8, y=A, logp=B, lse=B + 64, ent=None, ss=None):
        out = lp._Outputs(logp, lse, ent, ss)
        return L.lp_merge_shard_stats(stats, T, ctypes.byref(cp), y, ctypes.byref(out), None)

    assert merge(stats=None) == 1
    assert merge(y=None) == 1
    assert merge(lse=None) == 1
    assert merge(ss=B + 128) == 1                 # shard statistics are an input here, not an output
    assert merge(T=0, stats=None, y=None) == 0    # empty batch: no work
    assert merge() == 3                           # valid: fails only for want of a GPU

    def psum(parts=(A, A + 4096), n=None, count=1000, out=B, dtype=lp.LP_DTYPE_F32):
        P = (ctypes.c_void_p * max(len(parts), 1))(*parts)
        return L.lp_sum_partials(P, len(parts) if n is None else n, count, out, dtype, None)

    assert psum(n=0) == 1
    assert psum(n=65, parts=[A + 4096 * i for i in range(65)]) == 1
    assert psum(dtype=2) == 1
    assert psum(out=None) == 1
    assert psum(parts=(A + 4, A + 4096)) == 2     # misaligned part
    assert psum(out=B + 8) == 2                   # misaligned output
    assert psum(out=A + 4096) == 1                # output over a later part
    assert psum(out=A + 16) == 1                  # output over part 0, not exactly in place
    assert psum(out=A, dtype=lp.LP_DTYPE_BF16) == 1   # bf16 over fp32 part 0 is not in place
    assert psum(count=0, parts=(None,), out=None) == 0
    assert psum(out=A) == 3                       # in place into part 0: valid
    assert psum() == 3
