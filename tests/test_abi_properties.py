"""Property-based checks of the host-side validation and workspace sizing of the C ABI
(CPU only; the fake device pointers are never dereferenced because every call either
fails validation or stops at the device check, which fails without a GPU)."""
import ctypes

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


pytestmark = pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers; only safe without a GPU")


@pytest.fixture(scope="module")
def lp():
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    import lm_head_linear_tcgen05_gb300 as mod
    mod.lib()
    return mod


def _align(x, a=256):
    return (x + a - 1) // a * a


@st.composite
def partitions(draw):
    n = draw(st.integers(1, 8))
    widths = draw(st.lists(st.integers(0, 5000), min_size=n, max_size=n))
    vpad = sum(widths)
    if vpad == 0:
        widths[-1] = 1
        vpad = 1
    vreal = draw(st.integers(1, vpad))
    bounds = [0]
    for w in widths:
        bounds.append(bounds[-1] + w)
    return vreal, vpad, bounds


def _part(lp, vreal, vpad, bounds):
    return lp.VocabPartition(vreal, vpad, tuple((bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)))


@settings(max_examples=200, deadline=None)
@given(pt=partitions(), T=st.integers(0, 5000))
def test_forward_workspace_matches_layout(lp, pt, T):
    vreal, vpad, bounds = pt
    p = _part(lp, vreal, vpad, bounds)
    nb = 0
    for s, e in zip(bounds[:-1], bounds[1:]):
        real = max(min(e, vreal) - s, 0)
        nb += (real + 255) // 256
    expect = 3 * _align(nb * T * 4) + _align(T * 4)
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, T, 256, p) == expect
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD_FROM_LOGITS, T, 256, p) == 0
    assert lp.lp_workspace_size(lp.LP_OP_BACKWARD_FROM_LOGITS, T, 256, p) == 0


def _raw_partition(lp, vreal, vpad, ranges):
    arr = (lp._ShardRange * max(len(ranges), 1))(*[lp._ShardRange(s, e) for s, e in ranges])
    cp = lp._Partition(vreal, vpad, len(ranges), ctypes.cast(arr, ctypes.POINTER(lp._ShardRange)))
    return cp, arr


@st.composite
def broken_partitions(draw):
    """A valid partition with one mutation that makes it invalid."""
    vreal, vpad, bounds = draw(partitions())
    ranges = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    kinds = ["short", "long", "real_gt_pad", "real_zero", "too_many", "none"]
    if len(ranges) >= 2:
        kinds.append("hole")
        if ranges[1][0] >= 1:
            kinds.append("overlap")
    kind = draw(st.sampled_from(kinds))
    if kind == "hole":          # shard 1 starts one id after shard 0 ends
        ranges[1] = (ranges[1][0] + 1, ranges[1][1])
    elif kind == "overlap":     # shard 1 starts one id before shard 0 ends
        ranges[1] = (ranges[1][0] - 1, ranges[1][1])
    elif kind == "short":       # the shards stop before vocab_padded
        vpad += 1
    elif kind == "long":        # the shards run past vocab_padded
        vpad -= 1
    elif kind == "real_gt_pad":
        vreal = vpad + 1
    elif kind == "real_zero":
        vreal = 0
    elif kind == "too_many":
        ranges = [(i, i + 1) for i in range(9)]
        vreal, vpad = 9, 9
    else:
        ranges = []
    return vreal, vpad, ranges


@settings(max_examples=300, deadline=None)
@given(bp=broken_partitions(), T=st.integers(1, 3000))
def test_broken_partitions_are_rejected_before_any_launch(lp, bp, T):
    vreal, vpad, ranges = bp
    cp, keep = _raw_partition(lp, vreal, vpad, ranges)
    L = lp.lib()
    assert L.lp_workspace_size(lp.LP_OP_FORWARD, T, 256, ctypes.byref(cp)) == 0
    A = 0x100000
    Wa = (ctypes.c_void_p * max(len(ranges), 1))(*([A] * max(len(ranges), 1)))
    out = lp._Outputs(A, A, None, None)
    status = L.lp_forward(A, T, 256, Wa, None, ctypes.byref(cp), A, 0.7, ctypes.byref(out), A, 1 << 40, None)
    assert status == 1  # LP_ERR_INVALID_ARG, before the device is touched


@settings(max_examples=100, deadline=None)
@given(pt=partitions(), T=st.integers(1, 3000), H=st.sampled_from([8, 64, 4096, 65536]))
def test_valid_calls_reach_the_device_check(lp, pt, T, H):
    vreal, vpad, bounds = pt
    p = _part(lp, vreal, vpad, bounds)
    cp, keep = lp._c_partition(p)
    L = lp.lib()
    A = 0x100000
    n = len(bounds) - 1
    Wa = (ctypes.c_void_p * n)(*([A] * n))
    out = lp._Outputs(A, A, A, None)
    need = lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, p)
    assert L.lp_forward(A, T, H, Wa, None, ctypes.byref(cp), A, 0.7, ctypes.byref(out), A, need, None) == 3
    assert L.lp_forward(A, T, H, Wa, None, ctypes.byref(cp), A, 0.7, ctypes.byref(out), A, max(need, 1) - 1,
                        None) == (4 if need > 0 else 3)


@st.composite
def local_runs(draw):
    """A valid partition and one tensor-parallel rank's consecutive run of its shards."""
    vreal, vpad, bounds = draw(partitions())
    n = len(bounds) - 1
    k0 = draw(st.integers(0, n - 1))
    k1 = draw(st.integers(k0 + 1, n))
    return vreal, vpad, bounds, k0, k1


@settings(max_examples=200, deadline=None)
@given(lr=local_runs(), T=st.integers(0, 4000), mutate=st.sampled_from(["none", "hole", "past_end", "flag"]))
def test_rank_local_partitions(lp, lr, T, mutate):
    # a rank's run of shards, flagged local, is accepted and sized like those shards alone;
    # a gap inside it, an end past vocab_padded or a flag other than 0 / 1 is rejected
    vreal, vpad, bounds, k0, k1 = lr
    ranges = [(bounds[i], bounds[i + 1]) for i in range(k0, k1)]
    flag = 1
    if mutate == "hole" and len(ranges) >= 2:
        ranges[1] = (ranges[1][0] + 1, ranges[1][1] + 1)
    elif mutate == "past_end":
        ranges[-1] = (ranges[-1][0], vpad + 1)
    elif mutate == "flag":
        flag = 2
    else:
        mutate = "none"
    cp, keep = _raw_partition(lp, vreal, vpad, ranges)
    cp.local = flag
    got = lp.lib().lp_workspace_size(lp.LP_OP_FORWARD, T, 256, ctypes.byref(cp))
    if mutate != "none":
        assert got == 0
        return
    nb = sum((max(min(e, vreal) - s, 0) + 255) // 256 for s, e in ranges)
    assert got == 3 * _align(nb * T * 4) + _align(T * 4)
