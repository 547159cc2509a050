"""Vocabulary-parallel path on one GPU: each tensor-parallel rank's work is one call over a
rank-local partition (its own shards only); the ranks' per-shard statistics, gathered in
rank order and folded by lp_merge_shard_stats, must equal one call over every shard bit
for bit - for the fused forward, the logits-reuse forward and all three replay routes
(other ranks' replay ids and targets are skipped, not errors). The backward's dW and db
of a rank are bitwise those of the whole call, and its dX shares added in rank order by
lp_sum_partials give the whole dX (bitwise where the whole call splits its dX sum at the
same shard boundaries, as at the Qwen3-8B sharded size). Everything is also checked
against the fp64 oracle within the stated tolerances."""
import numpy as np
import pytest

import oracle
import synth
from lp_util import (TOL_ENT, TOL_GRAD_REL, TOL_LOGP, TOL_LSE, dev_bf16, dev_f32, dev_i32, dev_inputs, max_abs,
                     part_of, rel_fro)

pytestmark = pytest.mark.gpu


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


def _local(lp, part, ks):
    return lp.VocabPartition(part.vocab_real, part.vocab_padded, tuple(part.ranges[k] for k in ks), local=True)


def _same(a, b, keys):
    import torch
    for k in keys:
        assert torch.equal(a[k], b[k]), k


def _mask_from_ids(ids, ranges):
    masks = [np.zeros((ids.shape[0], e - s), np.uint8) for s, e in ranges]
    for t in range(ids.shape[0]):
        for v in ids[t]:
            for k, (s, e) in enumerate(ranges):
                if v >= 0 and s <= v < e:
                    masks[k][t, v - s] = 1
    return masks


CASES = [
    # (T, H, bounds, vocab_real, bias_std, rank -> shards)
    (700, 256, [0, 3000, 3000, 7000, 8192], 8000, 0.2, [[0, 1], [2], [3]]),   # empty shard, padding
    (130, 192, [0, 1000, 2000, 3000, 4096], 4090, None, [[0], [1, 2, 3]]),
]


@pytest.mark.parametrize("T,H,bounds,real,bias,ranks", CASES)
def test_rank_local_forward_and_replay_merge_to_the_whole_call(lp, T, H, bounds, real, bias, ranks):
    import torch
    part = synth.ranges_partition(real, bounds[-1], bounds)
    P = part_of(part)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=T, w_std=0.05, bias_std=bias)
    X, W, b, y = dev_inputs(inp)
    full = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    z = oracle.logits_from_bits(inp.X, inp.W, inp.bias, part, inp.tau)
    st = oracle.shard_stats(z, inp.y.astype(np.int64), part.ranges, part.vocab_real)
    stats = []
    for ks in ranks:
        Pl = _local(lp, part, ks)
        loc = lp.lp_forward(X, [W[k] for k in ks], None if b is None else [b[k] for k in ks], Pl, y, inp.tau,
                            shard_stats=True)
        assert lp.lp_get_device_error() == 0          # other ranks' targets are not errors
        stats.append(loc["shard_stats"])
        # the rank's own view: the softmax over its ids; logp -inf where y is another rank's
        lo, hi = part.ranges[ks[0]][0], part.ranges[ks[-1]][1]
        rl, rs, re = oracle.merge_shard_stats(np.stack([st[k].lse for k in ks]), np.stack([st[k].t for k in ks]),
                                              np.stack([st[k].h for k in ks]), inp.y, Pl.ranges, real)
        assert max_abs(_np(loc["lse"]), rs) <= TOL_LSE
        assert max_abs(_np(loc["entropy"]), re) <= TOL_ENT
        assert max_abs(_np(loc["logp"]), rl) <= TOL_LOGP
        here = (inp.y >= lo) & (inp.y < hi)
        assert np.all(np.isneginf(_np(loc["logp"])[~here]))
    gathered = torch.cat(stats)
    assert torch.equal(gathered, full["shard_stats"])
    merged = lp.lp_merge_shard_stats(gathered, y, P)
    assert lp.lp_get_device_error() == 0
    _same(merged, full, ("logp", "lse", "entropy"))
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    assert max_abs(_np(merged["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(merged["entropy"]), ref.entropy) <= TOL_ENT

    # logits reuse: each rank streams its own shards' logits
    L, yl, tau = synth.logits_inputs(T, part, 0.7, seed=T + 3)
    Ld = [dev_bf16(a) if a.shape[1] else None for a in L]
    yld = dev_i32(yl)
    full_l = lp.lp_forward_from_logits(Ld, P, yld, tau, shard_stats=True)
    stats = [lp.lp_forward_from_logits([Ld[k] for k in ks], _local(lp, part, ks), yld, tau,
                                       shard_stats=True)["shard_stats"] for ks in ranks]
    assert lp.lp_get_device_error() == 0
    gathered = torch.cat(stats)
    assert torch.equal(gathered, full_l["shard_stats"])
    _same(lp.lp_merge_shard_stats(gathered, yld, P), full_l, ("logp", "lse", "entropy"))
    ref_l = oracle.forward_from_logits(L, part, yl, tau)
    assert max_abs(_np(full_l["entropy"]), ref_l.entropy) <= TOL_ENT
    # the gradient with respect to the reused logits: each rank, given the merged LSE and
    # entropy, writes its own shards' gradient, bitwise the whole call's
    gl, hl = dev_f32(synth.upstream_grad(T, seed=T + 7)), dev_f32(synth.upstream_grad(T, seed=T + 8))
    whole_g = lp.lp_backward_from_logits(Ld, P, yld, tau, full_l["lse"], gl, entropy=full_l["entropy"],
                                         grad_entropy=hl, out_dtype=torch.float32)
    for ks in ranks:
        loc_g = lp.lp_backward_from_logits([Ld[k] for k in ks], _local(lp, part, ks), yld, tau, full_l["lse"], gl,
                                           entropy=full_l["entropy"], grad_entropy=hl, out_dtype=torch.float32)
        for j, k in enumerate(ks):
            assert (loc_g[j] is None) == (whole_g[k] is None)
            if whole_g[k] is not None:
                assert torch.equal(loc_g[j], whole_g[k]), k
    assert lp.lp_get_device_error() == 0

    # replay, all three routes; every rank gets every row's ids and skips the others' ones.
    # Some targets are made excluded ids (in a shard that keeps other ids, not in the set).
    ids, yr = synth.replay_ids(T, part, seed=T + 5)
    rng = np.random.default_rng(T)
    starts = [r[0] for r in part.ranges]
    for t in rng.choice(T, size=T // 5, replace=False):
        s, e = part.ranges[int(np.searchsorted(starts, yr[t], side="right") - 1)]
        kept = set(ids[t].tolist())
        cand = [v for v in range(s, min(e, real)) if v not in kept]
        if cand:
            yr[t] = cand[int(rng.integers(len(cand)))]
    ids_d, yr_d = dev_i32(ids), dev_i32(yr)
    masks = _mask_from_ids(ids, part.ranges)
    masks_d = [torch.from_numpy(m).cuda() if m.shape[1] else None for m in masks]
    routes = {
        "projection": (lambda Pp, ks: lp.lp_top_p_replay(X, [W[k] for k in ks], None if b is None else
                                                          [b[k] for k in ks], Pp, ids_d, yr_d, inp.tau,
                                                          shard_stats=True)),
        "logits": (lambda Pp, ks: lp.lp_top_p_replay_from_logits([Ld[k] for k in ks], Pp, ids_d, yr_d, tau,
                                                                 shard_stats=True)),
        "dense_mask": (lambda Pp, ks: lp.lp_top_p_replay_dense_mask(X, [W[k] for k in ks], None if b is None else
                                                                    [b[k] for k in ks], Pp, [masks_d[k] for k in ks],
                                                                    yr_d, inp.tau, shard_stats=True)),
    }
    ref_r = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, yr, inp.tau)
    for name, run in routes.items():
        whole = run(P, list(range(part.n_shards)))
        assert lp.lp_get_device_error() == 0, name
        gathered = torch.cat([run(_local(lp, part, ks), ks)["shard_stats"] for ks in ranks])
        assert lp.lp_get_device_error() == 0, name
        assert torch.equal(gathered, whole["shard_stats"]), name
        merged = lp.lp_merge_shard_stats(gathered, yr_d, P, entropy=False)
        _same(merged, whole, ("logp", "lse"))
        if name != "logits":
            assert max_abs(_np(merged["logp"]), ref_r.logp) <= TOL_LOGP, name
            assert max_abs(_np(merged["lse"]), ref_r.lse) <= TOL_LSE, name
            ss = _np(whole["shard_stats"])
            for k in range(part.n_shards):
                assert max_abs(ss[k, 1], ref_r.shard_t[k]) <= TOL_LOGP, name


def test_merge_entry_point_edge_rows(lp):
    """Hand-made statistics: a normal row, a row whose shards are all empty, a target in an
    empty shard, an excluded target (t = -inf), a target another call's partition holds
    (no shard of this partition), and a target outside the vocabulary (a device error)."""
    import torch
    part = synth.ranges_partition(90, 96, [0, 30, 60, 96])
    inf = np.inf
    lse = np.array([[1.5, -inf, -inf, 0.2, 0.3, 0.1],
                    [2.0, -inf, -inf, 0.4, 0.5, 0.2],
                    [0.7, -inf, 2.5, 0.6, -inf, 0.3]], np.float32)
    t = np.array([[0.9, 0.0, 0.0, -inf, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    h = np.array([[0.3, 0.0, 0.0, 0.5, 0.6, 0.7],
                  [1.1, 0.0, 0.8, 0.2, 0.9, 1.0],
                  [0.4, 0.0, 0.6, 0.1, 0.0, 0.3]], np.float32)
    y = np.array([5, 40, 35, 10, 70, 95], np.int32)      # row 5: 95 >= vocab_real 90
    stats = dev_f32(np.stack([lse, t, h], axis=1))       # [3, 3, 6]
    out = lp.lp_merge_shard_stats(stats, dev_i32(y), part_of(part))
    err = lp.lp_get_device_error()
    assert err == 5                                      # LP_ERR_TARGET_OUT_OF_RANGE (row 5)
    lg, ls, en = _np(out["logp"]), _np(out["lse"]), _np(out["entropy"])
    rl, rs, re = oracle.merge_shard_stats(lse, t, h, y, part.ranges, part.vocab_real)
    assert np.isneginf(ls[1]) and np.isneginf(lg[1]) and en[1] == 0.0       # every shard empty
    assert np.isneginf(lg[2])                            # y in shard 1, which is empty in row 2
    assert np.isneginf(lg[3])                            # excluded target
    assert np.isneginf(lg[4])                            # y = 70 in shard 2, empty in row 4
    assert np.isneginf(lg[5])
    assert not np.isnan(np.stack([lg, ls, en])).any()
    assert max_abs(lg[:5], rl[:5]) <= 1e-6 and max_abs(ls, rs) <= 1e-6 and max_abs(en, re) <= 1e-6
    # a partition that does not hold y: logp -inf, no error
    sub = lp.VocabPartition(90, 96, ((0, 30),), local=True)
    o2 = lp.lp_merge_shard_stats(stats[:1].contiguous(), dev_i32(np.full(6, 45, np.int32)), sub)
    assert lp.lp_get_device_error() == 0
    assert np.all(np.isneginf(_np(o2["logp"]))) and torch.equal(o2["lse"][:1], stats[0, 0, :1])


@pytest.mark.parametrize("n,count", [(1, 1003), (3, 4096), (5, 1003), (64, 37)])
def test_sum_partials_adds_in_rank_order(lp, n, count):
    import torch
    rng = np.random.default_rng(n * 1000 + count)
    parts = [(rng.standard_normal(count) * 10.0 ** float(rng.integers(-3, 4))).astype(np.float32) for _ in range(n)]
    expect = parts[0].copy()
    for q in parts[1:]:
        expect += q                                      # fp32, round to nearest, in order
    assert expect.dtype == np.float32
    d = [dev_f32(q) for q in parts]
    got = lp.lp_sum_partials(d)
    assert np.array_equal(_np(got), expect)
    got16 = lp.lp_sum_partials(d, out_dtype=torch.bfloat16)
    assert torch.equal(got16, torch.from_numpy(expect).to(torch.bfloat16).cuda())
    lp.lp_sum_partials(d, out=d[0])                      # in place into the first part
    assert np.array_equal(_np(d[0]), expect)


def test_rank_local_backward_matches_the_whole_call(lp):
    import torch
    T, H, bounds, real = 300, 128, [0, 3000, 3000, 7000, 8192], 8000
    ranks = [[0, 1], [2], [3]]
    part = synth.ranges_partition(real, bounds[-1], bounds)
    P = part_of(part)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=41, w_std=0.05, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    g = synth.upstream_grad(T, seed=41)
    hgrad = synth.upstream_grad(T, seed=42)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    gd, hd = dev_f32(g), dev_f32(hgrad)
    whole = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], gd, entropy=fwd["entropy"], grad_entropy=hd)
    shares = []
    for ks in ranks:
        loc = lp.lp_backward_ex(X, [W[k] for k in ks], [b[k] for k in ks], _local(lp, part, ks), y, inp.tau,
                                fwd["lse"], gd, entropy=fwd["entropy"], grad_entropy=hd)
        assert lp.lp_get_device_error() == 0
        for j, k in enumerate(ks):                       # a rank's dW and db are the whole call's
            if whole["dW"][k] is not None:
                assert torch.equal(loc["dW"][j], whole["dW"][k])
                assert torch.equal(loc["db"][j], whole["db"][k])
        shares.append(loc["dX"])
    dX = lp.lp_sum_partials(shares)
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, h=hgrad)
    assert rel_fro(_np(dX), ref.dX) <= TOL_GRAD_REL
    assert rel_fro(_np(dX), _np(whole["dX"])) <= 1e-5    # a different (fixed) order of the same sum
    again = lp.lp_sum_partials(shares)
    assert torch.equal(again, dX)


def test_vocab_parallel_at_the_sharded_qwen3_size(lp):
    """T=4096, H=4096, V=151936 padded to 152064 in 4 shards of 38016, bias: four one-shard
    ranks. Forward statistics merge to the 4-shard call bit for bit; the backward's dX
    shares added in rank order are the 4-shard call's dX bit for bit (its dX sum is split at
    the same shard boundaries), and each rank's dW, db are the whole call's."""
    import torch
    T, H, V, Vpad = 4096, 4096, 151936, 152064
    w4 = Vpad // 4
    part = synth.ranges_partition(V, Vpad, [0, w4, 2 * w4, 3 * w4, Vpad])
    P = part_of(part)
    X, W, b, y = synth.device_forward_inputs(T, H, part, 0.7, "cuda", seed=3, bias_std=0.01)
    tau = float(np.float32(0.7))
    g = torch.randn(T, generator=torch.Generator(device="cuda").manual_seed(3), device="cuda")
    full = lp.lp_forward(X, W, b, P, y, tau, shard_stats=True)
    stats = [lp.lp_forward(X, [W[k]], [b[k]], _local(lp, part, [k]), y, tau, shard_stats=True)["shard_stats"]
             for k in range(4)]
    gathered = torch.cat(stats)
    assert torch.equal(gathered, full["shard_stats"])
    _same(lp.lp_merge_shard_stats(gathered, y, P), full, ("logp", "lse", "entropy"))
    whole = lp.lp_backward(X, W, b, P, y, tau, full["lse"], g)
    shares = []
    for k in range(4):
        loc = lp.lp_backward(X, [W[k]], [b[k]], _local(lp, part, [k]), y, tau, full["lse"], g)
        assert torch.equal(loc["dW"][0], whole["dW"][k]) and torch.equal(loc["db"][0], whole["db"][k])
        shares.append(loc["dX"])
        del loc
    assert torch.equal(lp.lp_sum_partials(shares), whole["dX"])
    assert lp.lp_get_device_error() == 0
