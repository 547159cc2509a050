"""The bounds-checked build (liblp_debug.so: every index a kernel computes from the grid,
the partition, the targets or the replay ids is compared with its buffer's extent before
the access; a failed comparison records LP_ERR_BOUNDS and skips the access). It stands in
for a sanitizer's out-of-bounds checks.

Its self-test records LP_ERR_BOUNDS while the regular build's records nothing, and every
entry point run through it on ragged shapes (an empty shard, padded ids, H not a multiple
of 64, row strides wider than the rows) passes every check and returns the regular
build's bits."""
import numpy as np
import pytest

import synth
from lp_util import dev_bf16, dev_f32, dev_i32, dev_inputs, part_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    import torch
    from lm_head_linear_tcgen05_gb300 import _build
    regular = _build.build()
    debug = _build.build(debug_bounds=True)
    import lm_head_linear_tcgen05_gb300 as mod
    torch.cuda.set_device(0)
    yield mod, regular, debug
    mod.use_library(regular)          # later test modules run on the regular build


def test_bounds_selftest(libs):
    lp, regular, debug = libs
    lp.use_library(regular)
    assert not lp.lp_debug_bounds_build()
    lp.lp_selftest_bounds()
    assert lp.lp_get_device_error() == 0
    lp.use_library(debug)
    assert lp.lp_debug_bounds_build()
    lp.lp_selftest_bounds()
    assert lp.lp_get_device_error() == 10          # LP_ERR_BOUNDS, then cleared
    assert lp.lp_get_device_error() == 0
    lp.use_library(regular)


def _strided(t, extra=8):
    """A view of the 2-D tensor t whose row stride is t's width rounded up to 8, plus `extra`."""
    import torch
    T, w = t.shape
    buf = torch.zeros((T, (w + 7) // 8 * 8 + extra), dtype=t.dtype, device=t.device)
    buf[:, :w] = t
    return buf[:, :w]


def _every_entry_point(lp, case):
    import torch
    X, W, b, y, P, part, ids, masks, g, h, L, tau = case
    out = {}
    f = lp.lp_forward(X, W, b, P, y, tau, shard_stats=True)
    out.update({f"fwd_{k}": v for k, v in f.items() if v is not None})
    fl = lp.lp_forward_from_logits(L, P, y, tau, shard_stats=True)
    out.update({f"logits_{k}": v for k, v in fl.items() if v is not None})
    r = lp.lp_top_p_replay(X, W, b, P, ids, y, tau, shard_stats=True)
    out.update({f"replay_{k}": v for k, v in r.items() if v is not None})
    rl = lp.lp_top_p_replay_from_logits(L, P, ids, y, tau, shard_stats=True)
    out.update({f"replay_logits_{k}": v for k, v in rl.items() if v is not None})
    dm = lp.lp_top_p_replay_dense_mask(X, W, b, P, masks, y, tau, shard_stats=True)
    out.update({f"mask_{k}": v for k, v in dm.items() if v is not None})
    bw = lp.lp_backward(X, W, b, P, y, tau, f["lse"], g, entropy=f["entropy"], grad_entropy=h)
    out["dX"] = bw["dX"]
    for k, (dw, db) in enumerate(zip(bw["dW"], bw["db"])):
        if dw is not None:
            out[f"dW{k}"], out[f"db{k}"] = dw, db
    dL = lp.lp_backward_from_logits(L, P, y, tau, fl["lse"], g, entropy=fl["entropy"], grad_entropy=h,
                                    out_dtype=torch.float32)
    for k, d in enumerate(dL):
        if d is not None:
            out[f"dL{k}"] = d
    # the vocabulary-parallel steps: a rank-local replay (other ranks' ids skipped), the
    # rank-ordered merge of statistics and the ordered sum of partials
    ranges = P.ranges
    Pl = lp.VocabPartition(P.vocab_real, P.vocab_padded, ranges[2:], local=True)
    rloc = lp.lp_top_p_replay(X, W[2:], None if b is None else b[2:], Pl, ids, y, tau, shard_stats=True)
    out.update({f"replay_local_{k}": v for k, v in rloc.items() if v is not None})
    m = lp.lp_merge_shard_stats(f["shard_stats"], y, P)
    out.update({f"merge_{k}": v for k, v in m.items() if v is not None})
    out["sum"] = lp.lp_sum_partials([bw["dX"], bw["dX"].flip(0).contiguous(), bw["dX"]])
    torch.cuda.synchronize()
    return out


def test_every_entry_point_passes_the_bounds_checks(libs):
    import torch
    lp, regular, debug = libs
    bounds, real = [0, 3000, 3000, 8000, 8192], 8100            # an empty shard and 92 padded ids
    part = synth.ranges_partition(real, bounds[-1], bounds)
    T, H = 77, 136
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=21, w_std=0.05, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    ids, _ = synth.replay_ids(T, part, seed=22)
    masks = []
    for k, (s, e) in enumerate(part.ranges):
        m = np.zeros((T, e - s), np.uint8)
        for t in range(T):
            for v in ids[t]:
                if s <= v < e:
                    m[t, v - s] = 1
        masks.append(torch.from_numpy(m).cuda() if e > s else None)
    Lh, _, _ = synth.logits_inputs(T, part, 0.7, seed=23)
    L = [_strided(dev_bf16(a)) if a.shape[1] else None for a in Lh]
    case = (X, W, b, y, part_of(part), part, dev_i32(ids), masks, dev_f32(synth.upstream_grad(T, seed=24)),
            dev_f32(synth.upstream_grad(T, seed=25)), L, inp.tau)
    lp.use_library(regular)
    ref = _every_entry_point(lp, case)
    assert lp.lp_get_device_error() == 0
    lp.use_library(debug)
    got = _every_entry_point(lp, case)
    assert lp.lp_get_device_error() == 0           # no check failed
    lp.use_library(regular)
    for key, v in ref.items():
        assert torch.equal(got[key], v), key
