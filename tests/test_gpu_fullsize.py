"""Parity at the full benchmark sizes, in the launch configuration bench.py times, on
sampled rows the oracle computes one by one (plus properties that hold at any size):

* Qwen3-8B-shaped forward: T=4096, H=4096, V=151936, tau=0.7; 1 x 4096 vs 8 x 512 bitwise;
* vocabulary-sharded forward + backward: V=151936 padded to 152064 in 4 shards of 38016,
  bias; dX on sampled rows at T=4096, dW/db on sampled vocabulary rows at T'=256;
* logits reuse: T=8192 x 151936 bf16 logits, 1 % peaked rows (and T=2048 in the 4 padded
  shards of the sharded layout);
* compact top-p replay: T=8192, 4 shards of 37984, 1-64 ids per row, 25 % of rows with an
  empty shard; dense keep-mask route bitwise equal.
"""
import numpy as np
import pytest

import oracle
import synth
from lp_util import (TOL_ENT, TOL_GRAD_REL, TOL_LOGP, TOL_LSE, dev_bf16, dev_f32, dev_i32, dev_inputs, max_abs,
                     part_of, rel_fro)

pytestmark = pytest.mark.gpu

T2, H, V = 4096, 4096, 151936
TAU = 0.7


@pytest.fixture(scope="module")
def lp():
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    import lm_head_linear_tcgen05_gb300 as mod
    import torch
    assert mod.lp_device_supported()
    torch.cuda.set_device(0)
    return mod


def _np(t):
    return t.detach().cpu().numpy()


def _sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, T // 2, T - 129, T - 128, T - 1]
    rest = rng.choice(T, size=n - len(fixed), replace=False)
    return np.unique(np.concatenate([fixed, rest]))


def test_qwen3_8b_forward_sampled_rows_and_batch_invariance(lp):
    import torch
    part = synth.even_partition(V, 1)
    inp = synth.forward_inputs(T2, H, part, tau=TAU, seed=0)
    X, W, _, y = dev_inputs(inp)
    P = part_of(part)
    out = lp.lp_forward(X, W, None, P, y, inp.tau)          # one call over all 4096 rows
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T2, 64, 1)
    ref = oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"])[rows], ref.entropy) <= TOL_ENT
    # every row: entropy in [0, log V], logp <= 0, no NaN
    lg, en = _np(out["logp"]), _np(out["entropy"])
    assert np.all(lg <= 0) and np.all(np.isfinite(lg))
    assert np.all(en >= 0) and np.all(en <= np.log(V) + 1e-4)
    # 8 batches of 512 rows give the same bits
    for s in range(0, T2, 512):
        o = lp.lp_forward(X[s:s + 512].contiguous(), W, None, P, y[s:s + 512].contiguous(), inp.tau)
        for k in ("logp", "lse", "entropy"):
            assert torch.equal(o[k], out[k][s:s + 512]), (s, k)


def _sharded():
    part = synth.ranges_partition(V, 152064, [0, 38016, 76032, 114048, 152064])
    return part


def test_sharded_forward_and_backward_dx_sampled_rows(lp):
    part = _sharded()
    inp = synth.forward_inputs(T2, H, part, tau=TAU, seed=3, bias_std=0.01)
    g = synth.upstream_grad(T2, seed=3)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T2, 24, 2)
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, rows=rows)
    assert max_abs(_np(fwd["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(fwd["lse"])[rows], ref.lse) <= TOL_LSE
    assert max_abs(_np(fwd["entropy"])[rows], ref.entropy) <= TOL_ENT
    ss = _np(fwd["shard_stats"])
    for k, s in enumerate(ref.shards):
        assert max_abs(ss[k, 0][rows], s.lse) <= TOL_LSE
        assert max_abs(ss[k, 1][rows], s.t) <= TOL_LOGP
    dx_rows = rows[:8]
    dX, _, _ = oracle.backward_sampled(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, dx_rows, [[], [], [], []])
    assert rel_fro(_np(bw["dX"])[dx_rows], dX) <= TOL_GRAD_REL
    # properties at full size: sum_v db_v = sum_t g_t (1 - sum_v p_tv) / tau = 0, and
    # the 128 padded ids of the last shard get exactly zero gradient
    total = sum(float(_np(d).astype(np.float64).sum()) for d in bw["db"])
    scale = float(np.abs(g).sum()) / TAU
    assert abs(total) <= 1e-3 * scale
    assert np.all(_np(bw["dW"][3])[37888:] == 0) and np.all(_np(bw["db"][3])[37888:] == 0)


def test_sharded_backward_dw_db_sampled_vocab_rows_short_batch(lp):
    part = _sharded()
    T = 256
    inp = synth.forward_inputs(T, H, part, tau=TAU, seed=5, bias_std=0.01)
    g = synth.upstream_grad(T, seed=5)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0
    rng = np.random.default_rng(7)
    dw_rows = []
    for k, (s, e) in enumerate(part.ranges):
        r = list(rng.choice(e - s, size=12, replace=False)) + [0, min(e, V) - s - 1]
        # the rows that hold some targets carry the one-hot term
        r += [int(t) - s for t in inp.y[:3] if s <= t < e]
        if k == 3:
            r += [37888, 38015]                      # padded ids
        dw_rows.append(np.unique(np.array(r, dtype=np.int64)))
    dX, dW, db = oracle.backward_sampled(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, np.arange(8), dw_rows)
    assert rel_fro(_np(bw["dX"])[:8], dX) <= TOL_GRAD_REL
    for k in range(4):
        assert rel_fro(_np(bw["dW"][k])[dw_rows[k]], dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(_np(bw["db"][k])[dw_rows[k]], db[k]) <= TOL_GRAD_REL, k


def test_logits_reuse_full_size_sampled_rows(lp):
    import torch
    part = synth.even_partition(V, 1)
    T = 8192
    L, y, tau = synth.logits_inputs(T, part, TAU, seed=4)
    Ld = [dev_bf16(L[0])]
    out = lp.lp_forward_from_logits(Ld, part_of(part), dev_i32(y), tau)
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T, 512, 3)
    ref = oracle.forward_from_logits(L, part, y, tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"])[rows], ref.entropy) <= TOL_ENT
    again = lp.lp_forward_from_logits(Ld, part_of(part), dev_i32(y), tau)
    assert torch.equal(again["lse"], out["lse"]) and torch.equal(again["entropy"], out["entropy"])


def test_logits_reuse_full_width_four_padded_shards(lp):
    """The sharded layout (4 x 38016 ids, the last 128 of them padding) at full width: every
    shard ends in a partial batch of vectors, and per-shard results are merged at the end of
    the row. Sampled rows against the oracle, shard statistics included; rows computed in a
    smaller batch keep their bits."""
    import torch
    part = _sharded()
    T = 2048
    L, y, tau = synth.logits_inputs(T, part, TAU, seed=44)
    Ld = [dev_bf16(a) for a in L]
    out = lp.lp_forward_from_logits(Ld, part_of(part), dev_i32(y), tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T, 256, 5)
    ref = oracle.forward_from_logits(L, part, y, tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"])[rows], ref.entropy) <= TOL_ENT
    ss = _np(out["shard_stats"])
    for k, s in enumerate(ref.shards):
        assert max_abs(ss[k, 0][rows], s.lse) <= TOL_LSE
        assert max_abs(ss[k, 1][rows], s.t) <= TOL_LOGP
        assert max_abs(ss[k, 2][rows], s.h) <= TOL_ENT
    sub = lp.lp_forward_from_logits([x[1000:1100] for x in Ld], part_of(part), dev_i32(y[1000:1100]), tau)
    for key in ("logp", "lse", "entropy"):
        assert torch.equal(sub[key], out[key][1000:1100])


def test_replay_full_size_and_dense_mask(lp):
    import torch
    part = synth.even_partition(V, 4)
    T = 8192
    inp = synth.forward_inputs(T, H, part, tau=TAU, seed=5)
    ids, y = synth.replay_ids(T, part, seed=5)
    X, W, _, _ = dev_inputs(inp)
    P = part_of(part)
    ids_d, y_d = dev_i32(ids), dev_i32(y)
    out = lp.lp_top_p_replay(X, W, None, P, ids_d, y_d, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T, 1024, 4)
    ref = oracle.top_p_replay(inp.X, inp.W, None, part, ids, y, inp.tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    ss = _np(out["shard_stats"])
    for k in range(4):
        assert max_abs(ss[k, 0][rows], ref.shard_lse[k]) <= TOL_LSE
        assert max_abs(ss[k, 1][rows], ref.shard_t[k]) <= TOL_LOGP
    # rows with an empty shard report -inf there and stay NaN-free
    assert np.isneginf(ss[:, 0]).any() and not np.isnan(ss).any()
    # the dense keep-mask route over full-width masks gives the same bits
    masks = []
    for k, (s, e) in enumerate(part.ranges):
        m = torch.zeros((T, e - s), dtype=torch.uint8, device="cuda")
        sel = (ids_d >= s) & (ids_d < e)
        r = torch.arange(T, device="cuda").unsqueeze(1).expand_as(ids_d)[sel]
        m[r.long(), (ids_d[sel] - s).long()] = 1
        masks.append(m)
    dm = lp.lp_top_p_replay_dense_mask(X, W, None, P, masks, y_d, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    for k in ("logp", "lse", "shard_stats"):
        assert torch.equal(dm[k], out[k]), k


def test_replay_from_logits_full_size(lp):
    import torch
    part = synth.even_partition(V, 4)
    T = 8192
    L, _, tau = synth.logits_inputs(T, part, TAU, seed=6)
    ids, y = synth.replay_ids(T, part, seed=6)
    Ld = [dev_bf16(a) for a in L]
    out = lp.lp_top_p_replay_from_logits(Ld, part_of(part), dev_i32(ids), dev_i32(y), tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T, 1024, 5)
    ref = oracle.top_p_replay_from_logits(L, part, ids, y, tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    ss = _np(out["shard_stats"])
    for k in range(4):
        assert max_abs(ss[k, 0][rows], ref.shard_lse[k]) <= TOL_LSE


@pytest.mark.parametrize("T,Hh,Vv,shards", [(2048, 8192, 128256, 2), (1024, 2048, 262144 - 517, 4)])
def test_other_lm_head_shapes_sampled_rows(lp, T, Hh, Vv, shards):
    # larger hidden size with a 128256-id vocabulary in two shards, and a wide vocabulary whose
    # size is not a multiple of any tile (padded to split evenly): sampled rows against the
    # oracle, the backward's dX on a few rows, and batch invariance on a row slice
    import torch
    Vpad = -(-Vv // (shards * 64)) * shards * 64
    w = Vpad // shards
    part = synth.ranges_partition(Vv, Vpad, [k * w for k in range(shards + 1)])
    inp = synth.forward_inputs(T, Hh, part, tau=0.9, seed=T + Hh, w_std=0.02, bias_std=0.01)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    out = lp.lp_forward(X, W, b, P, y, inp.tau)
    assert lp.lp_get_device_error() == 0
    rows = _sample_rows(T, 24, Hh)
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, rows=rows)
    assert max_abs(_np(out["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"])[rows], ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"])[rows], ref.entropy) <= TOL_ENT
    sl = lp.lp_forward(X[100:612].contiguous(), W, b, P, y[100:612].contiguous(), inp.tau)
    assert torch.equal(sl["logp"], out["logp"][100:612]) and torch.equal(sl["entropy"], out["entropy"][100:612])
    g = synth.upstream_grad(T, seed=Hh)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, out["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0
    dx_rows = rows[:6]
    dX, _, _ = oracle.backward_sampled(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, dx_rows, [[]] * shards)
    assert rel_fro(_np(bw["dX"])[dx_rows], dX) <= TOL_GRAD_REL
