"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here reuses the oracle's own formulas: each check is a closed form, a
library routine on a special case, an invariant, a brute force written
independently (pure Python, its own bf16 decode, math.fsum), or a finite
difference.
"""
import json
import math
import os
import struct

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dec(bits):
    """bf16 bits -> Python float, independent of the oracle's decoder."""
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def test_bf16_decode_against_the_format_definition():
    # bf16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits; value written out from
    # the definition for every one of the 65536 codes (normal, subnormal, zero, inf, NaN)
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # signalling NaN codes widen with a warning
        got = oracle.bf16_to_f64(codes)
    for c in range(1 << 16):
        s, e, f = c >> 15, (c >> 7) & 0xFF, c & 0x7F
        sign = -1.0 if s else 1.0
        if e == 0xFF:
            if f == 0:
                assert got[c] == sign * math.inf, hex(c)
            else:
                assert math.isnan(got[c]), hex(c)
            continue
        want = sign * (math.ldexp(f, -126 - 7) if e == 0 else math.ldexp(128 + f, e - 127 - 7))
        assert got[c] == want and math.copysign(1.0, got[c]) == sign, hex(c)


def _zeros_like_W(part, H):
    return [np.zeros((e - s, H), np.uint16) for s, e in part.ranges]


def _bias_bits(vals):
    return synth.bf16_bits(np.asarray(vals, np.float32))


# ---------------------------------------------------------------- closed forms

def test_w_zero_gives_uniform_over_real_vocab_with_padding():
    # z == 0 on the real ids: logp = -log V_real, LSE = entropy = log V_real.
    # With 24 padded ids, -log(1024) would differ from -log(1000) by 0.0237.
    part = synth.even_partition(1000, 4, vocab_padded=1024)
    T, H = 5, 16
    rng = np.random.default_rng(0)
    X = synth.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    y = rng.integers(0, 1000, T).astype(np.int32)
    r = oracle.forward(X, _zeros_like_W(part, H), None, part, y, 0.7)
    np.testing.assert_allclose(r.logp, -math.log(1000), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.lse, math.log(1000), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.entropy, math.log(1000), rtol=0, atol=1e-12)


def test_constant_bias_shifts_lse_by_c_over_tau():
    part = synth.even_partition(96, 3)
    T, H, c, tau = 3, 8, 1.5, 0.75
    b = [_bias_bits(np.full(32, c)) for _ in range(3)]
    X = np.zeros((T, H), np.uint16)
    y = np.array([0, 50, 95], np.int32)
    r = oracle.forward(X, _zeros_like_W(part, H), b, part, y, tau)
    np.testing.assert_allclose(r.lse, c / tau + math.log(96), atol=1e-12)
    np.testing.assert_allclose(r.logp, -math.log(96), atol=1e-12)


def test_two_level_logits_closed_form():
    # k ids at alpha = b/tau, the rest at 0:
    # LSE = log(k e^a + V - k); entropy = LSE - k a e^a / Z.
    V, k, tau, bval = 200, 7, 0.5, 2.0
    alpha = bval / tau
    part = synth.even_partition(V, 2)
    hot = np.zeros(V, np.float32)
    hot[[3, 17, 99, 100, 150, 151, 199]] = bval
    b = [_bias_bits(hot[:100]), _bias_bits(hot[100:])]
    X = np.zeros((2, 4), np.uint16)
    y = np.array([17, 5], np.int32)
    r = oracle.forward(X, _zeros_like_W(part, 4), b, part, y, tau)
    Z = k * math.exp(alpha) + (V - k)
    lse = math.log(Z)
    ent = lse - k * alpha * math.exp(alpha) / Z
    np.testing.assert_allclose(r.lse, lse, atol=1e-12)
    np.testing.assert_allclose(r.entropy, ent, atol=1e-12)
    np.testing.assert_allclose(r.logp, [alpha - lse, -lse], atol=1e-12)


def test_one_dominant_logit_gives_logp_zero_entropy_zero():
    # z_y = 1000, the other 63 ids 0: exp(-1000) underflows, so LSE = 1000,
    # logp = 0 and entropy = 0 exactly in float64
    V, tau = 64, 1.0
    part = synth.even_partition(V, 1)
    hot = np.zeros(V, np.float32)
    hot[11] = 1000.0                       # exactly representable in bf16
    X = np.zeros((1, 8), np.uint16)
    r = oracle.forward(X, _zeros_like_W(part, 8), [_bias_bits(hot)], part,
                       np.array([11], np.int32), tau)
    assert r.logp[0] == 0.0
    assert abs(r.entropy[0]) < 1e-12
    assert r.lse[0] == 1000.0


def test_empty_shard_convention_printed_on_the_pages():
    # tests/golden/empty_shard.json holds the values the replay page prints for a
    # vocabulary shard with no candidates
    with open(os.path.join(GOLDEN, "empty_shard.json")) as f:
        gold = json.load(f)["local"]
    part = synth.ranges_partition(40, 48, [0, 16, 32, 48])
    inp = synth.forward_inputs(2, 8, part, tau=0.7, seed=0, w_std=0.3)
    ids = np.full((2, 64), -1, np.int32)
    ids[0, :3] = [1, 2, 20]                  # shard 2 ([32,48)) empty in row 0
    ids[1, :2] = [35, 36]                    # shards 0 and 1 empty in row 1
    y = np.array([20, 35], np.int32)
    rep = oracle.top_p_replay(inp.X, inp.W, None, part, ids, y, inp.tau)
    for k, t in [(2, 0), (0, 1), (1, 1)]:
        assert rep.shard_lse[k, t] == float(gold["lse"])
        assert rep.shard_t[k, t] == gold["target_logit"]
    # the dense path: a shard made only of padding ids is empty too
    part2 = synth.ranges_partition(32, 48, [0, 16, 32, 48])
    r = oracle.forward(inp.X, inp.W, None, part2, np.array([3, 17], np.int32), inp.tau)
    assert np.all(r.shards[2].lse == float(gold["lse"]))
    assert np.all(r.shards[2].t == gold["target_logit"])


@pytest.mark.parametrize("V,k,tau,bval", [(50, 1, 1.0, 3.0), (1000, 10, 0.7, 0.5), (7, 6, 2.0, -4.0)])
def test_two_level_closed_form_parametrized(V, k, tau, bval):
    part = synth.even_partition(V, 1)
    hot = np.zeros(V, np.float32)
    hot[:k] = bval
    X = np.zeros((1, 4), np.uint16)
    r = oracle.forward(X, _zeros_like_W(part, 4), [_bias_bits(hot)], part, np.array([V - 1], np.int32), tau)
    a = bval / tau                          # bval is exactly representable in bf16
    Z = k * math.exp(a) + (V - k)
    lse = math.log(Z)
    np.testing.assert_allclose(r.lse[0], lse, atol=1e-12)
    np.testing.assert_allclose(r.logp[0], -lse, atol=1e-12)
    np.testing.assert_allclose(r.entropy[0], lse - k * a * math.exp(a) / Z, atol=1e-12)


# ------------------------------------------------------- library special case

def test_matches_torch_log_softmax_float64():
    torch = pytest.importorskip("torch")
    part = synth.ranges_partition(300, 320, [0, 100, 100, 250, 320])   # one empty shard
    inp = synth.forward_inputs(6, 24, part, tau=0.7, seed=3, w_std=0.3, bias_std=0.5)
    r = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    X = torch.from_numpy(oracle.bf16_to_f64(inp.X))
    W = torch.cat([torch.from_numpy(oracle.bf16_to_f64(w)) for w in inp.W])[:300]
    b = torch.cat([torch.from_numpy(oracle.bf16_to_f64(x)) for x in inp.bias])[:300]
    z = (X @ W.T + b) / inp.tau
    ls = torch.log_softmax(z, dim=1)
    ref_logp = ls[torch.arange(6), torch.from_numpy(inp.y.astype(np.int64))].numpy()
    ref_lse = torch.logsumexp(z, dim=1).numpy()
    ref_ent = -(ls.exp() * ls).sum(dim=1).numpy()
    np.testing.assert_allclose(r.logp, ref_logp, atol=1e-11)
    np.testing.assert_allclose(r.lse, ref_lse, atol=1e-11)
    np.testing.assert_allclose(r.entropy, ref_ent, atol=1e-11)


# ------------------------------------------------------------------ brute force

def _brute(X, W, b, part, y, tau):
    """Pure-Python forward with math.fsum; returns lists logp, lse, entropy."""
    out = []
    for t in range(len(y)):
        zs = {}
        for k, (vs, ve) in enumerate(part.ranges):
            for j in range(ve - vs):
                v = vs + j
                if v >= part.vocab_real:
                    continue
                a = math.fsum(_dec(X[t][h]) * _dec(W[k][j][h]) for h in range(len(X[t])))
                if b is not None:
                    a += _dec(b[k][j])
                zs[v] = a / tau
        M = max(zs.values())
        lse = M + math.log(math.fsum(math.exp(z - M) for z in zs.values()))
        ent = -math.fsum(math.exp(z - lse) * (z - lse) for z in zs.values())
        out.append((zs[int(y[t])] - lse, lse, ent))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_tiny_multishard_padded(seed):
    part = synth.ranges_partition(50, 64, [0, 13, 13, 40, 64])
    inp = synth.forward_inputs(4, 16, part, tau=0.7, seed=seed, w_std=0.4, bias_std=0.3)
    r = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    ref = _brute(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    np.testing.assert_allclose(r.logp, [o[0] for o in ref], atol=1e-12)
    np.testing.assert_allclose(r.lse, [o[1] for o in ref], atol=1e-12)
    np.testing.assert_allclose(r.entropy, [o[2] for o in ref], atol=1e-12)


def test_brute_force_logits_reuse_applies_tau_once():
    part = synth.ranges_partition(40, 48, [0, 20, 48])
    L, y, tau = synth.logits_inputs(3, part, 0.7, seed=5, peak_frac=0.1)
    r = oracle.forward_from_logits(L, part, y, tau)
    for t in range(3):
        zs = []
        for k, (vs, ve) in enumerate(part.ranges):
            for j in range(ve - vs):
                if vs + j < 40:
                    zs.append(_dec(L[k][t][j]) / tau)
        M = max(zs)
        lse = M + math.log(math.fsum(math.exp(z - M) for z in zs))
        assert abs(r.lse[t] - lse) < 1e-12
        assert abs(r.logp[t] - (zs[int(y[t])] - lse)) < 1e-12
        ent = -math.fsum(math.exp(z - lse) * (z - lse) for z in zs)
        assert abs(r.entropy[t] - ent) < 1e-12


# ------------------------------------------------------------------------ merge

def test_merge_of_shards_equals_unsharded():
    part = synth.ranges_partition(500, 512, [0, 100, 100, 300, 499, 512])  # empty + tiny shards
    inp = synth.forward_inputs(8, 32, part, tau=0.6, seed=9, w_std=0.2, bias_std=0.2)
    r = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    logp, lse, ent = oracle.merge_shards(r.shards, inp.y.astype(np.int64), part.ranges)
    np.testing.assert_allclose(logp, r.logp, atol=1e-12)
    np.testing.assert_allclose(lse, r.lse, atol=1e-12)
    np.testing.assert_allclose(ent, r.entropy, atol=1e-12)
    # the empty shard [100,100) and the all-padding shard [499..512) minus id 499
    assert np.all(np.isneginf(r.shards[1].lse))
    assert np.all(r.shards[1].t == 0) and np.all(r.shards[1].h == 0)


def test_merge_all_empty_row_convention():
    st = [oracle.ShardStats(np.array([-np.inf]), np.zeros(1), np.zeros(1)) for _ in range(3)]
    logp, lse, ent = oracle.merge_shards(st, np.array([5]), ((0, 4), (4, 8), (8, 12)))
    assert np.isneginf(lse[0]) and np.isneginf(logp[0]) and ent[0] == 0.0


def test_merged_replay_statistics_reproduce_the_replay():
    # the replay's per-shard (lse, t) exchanged and merged give the replay's own logp and
    # LSE, computed directly over each row's set: target found, target excluded from a
    # non-empty shard (t = -inf), target in an empty shard (lse = -inf, t = 0)
    part = synth.ranges_partition(60, 64, [0, 20, 40, 64])
    inp = synth.forward_inputs(4, 16, part, tau=0.7, seed=6, w_std=0.3, bias_std=0.1)
    ids = np.full((4, 64), -1, np.int32)
    ids[0, :4] = [3, 25, 41, 59]
    ids[1, :3] = [3, 25, 41]
    ids[2, :2] = [25, 41]
    ids[3, :2] = [1, 2]
    y = np.array([25, 5, 7, 45], np.int32)   # found; excluded from shard 0; shard 0 empty; shard 2 empty
    rep = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, y, inp.tau)
    assert rep.shard_t[0, 1] == -np.inf and np.isfinite(rep.shard_lse[0, 1])
    assert rep.shard_t[0, 2] == 0.0 and np.isneginf(rep.shard_lse[0, 2])
    logp, lse, _ = oracle.merge_shard_stats(rep.shard_lse, rep.shard_t, np.zeros_like(rep.shard_t), y,
                                            part.ranges, part.vocab_real)
    np.testing.assert_array_equal(np.isneginf(logp), [False, True, True, True])
    assert abs(logp[0] - rep.logp[0]) < 1e-12
    np.testing.assert_allclose(lse, rep.lse, atol=1e-12)


def test_shard_entropy_two_level_closed_form():
    # inside one shard of n real ids (padding excluded), k ids at alpha and the rest at 0:
    # h = log(k e^a + n - k) - k a e^a / (k e^a + n - k)
    part = synth.ranges_partition(30, 32, [0, 10, 32])
    n, k, alpha = 20, 3, 1.7                             # shard 1 holds real ids [10, 30)
    z = np.zeros((1, 30))
    z[0, 10:10 + k] = alpha
    st = oracle.shard_stats(z, np.array([12]), part.ranges, 30)
    Z = k * math.exp(alpha) + n - k
    assert abs(st[1].h[0] - (math.log(Z) - k * alpha * math.exp(alpha) / Z)) < 1e-12
    assert abs(st[0].h[0] - math.log(10)) < 1e-12      # uniform shard: log n


def test_merge_of_a_subset_of_shards_is_the_subsets_own_softmax():
    # what one tensor-parallel rank sees: the merge of its own shards only is the softmax
    # over its ids; a target held by another rank gives logp = -inf there
    part = synth.ranges_partition(500, 512, [0, 100, 250, 380, 512])
    inp = synth.forward_inputs(6, 32, part, tau=0.6, seed=9, w_std=0.2, bias_std=0.2)
    z = oracle.logits_from_bits(inp.X, inp.W, inp.bias, part, inp.tau)
    y = inp.y.astype(np.int64)
    y[:3] = [120, 300, 10]
    st = oracle.shard_stats(z, y, part.ranges, part.vocab_real)
    sub = [1, 2]                                         # this rank holds [100, 380)
    logp, lse, ent = oracle.merge_shard_stats(np.stack([st[k].lse for k in sub]), np.stack([st[k].t for k in sub]),
                                              np.stack([st[k].h for k in sub]), y,
                                              [part.ranges[k] for k in sub], part.vocab_real)
    lz, ll, le = oracle.dense_stats(z[:, 100:380], np.clip(y - 100, 0, 279))
    np.testing.assert_allclose(lse, ll, atol=1e-12)
    np.testing.assert_allclose(ent, le, atol=1e-12)
    local = (y >= 100) & (y < 380)
    np.testing.assert_allclose(logp[local], lz[local], atol=1e-12)
    assert np.all(np.isneginf(logp[~local]))


def test_shard_stats_match_local_closed_form():
    # shard local LSE with z == 0: log(#real ids in shard)
    part = synth.ranges_partition(90, 96, [0, 30, 60, 96])
    X = np.zeros((2, 4), np.uint16)
    r = oracle.forward(X, _zeros_like_W(part, 4), None, part, np.array([1, 70], np.int32), 0.7)
    np.testing.assert_allclose([s.lse[0] for s in r.shards], np.log([30, 30, 30]), atol=1e-12)


# ----------------------------------------------------------------------- replay

def _full_set_ids(T, V):
    ids = np.full((T, 64), -1, np.int32)
    for t in range(T):
        ids[t, :V] = np.random.default_rng(t).permutation(V)
    return ids


def test_replay_with_whole_vocab_equals_dense():
    part = synth.ranges_partition(60, 64, [0, 16, 32, 48, 64])
    inp = synth.forward_inputs(5, 32, part, tau=0.7, seed=4, w_std=0.3, bias_std=0.2)
    ids = _full_set_ids(5, 60)
    dense = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    rep = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, inp.y, inp.tau)
    np.testing.assert_allclose(rep.lse, dense.lse, atol=1e-12)
    np.testing.assert_allclose(rep.logp, dense.logp, atol=1e-12)
    for k in range(4):
        np.testing.assert_allclose(rep.shard_lse[k], dense.shards[k].lse, atol=1e-12)
        np.testing.assert_allclose(rep.shard_t[k], dense.shards[k].t, atol=1e-12)


def test_replay_single_id_and_missing_target():
    part = synth.even_partition(100, 2)
    inp = synth.forward_inputs(2, 16, part, tau=0.7, seed=1, w_std=0.3)
    ids = np.full((2, 64), -1, np.int32)
    ids[0, [5, 9, 40]] = 77                  # one distinct id, duplicated
    ids[1, 0] = 3
    y = np.array([77, 4], np.int32)          # row 1's target is not in its set
    rep = oracle.top_p_replay(inp.X, inp.W, None, part, ids, y, inp.tau)
    z77 = math.fsum(_dec(inp.X[0][h]) * _dec(inp.W[1][27][h]) for h in range(16)) / inp.tau
    assert rep.logp[0] == 0.0
    assert abs(rep.lse[0] - z77) < 1e-12
    assert np.isneginf(rep.logp[1]) and np.isfinite(rep.lse[1])
    assert np.isneginf(rep.shard_lse[0, 0]) and rep.shard_t[0, 0] == 0.0   # empty shard 0 in row 0


def test_replay_invariant_to_slot_order_and_duplicates():
    part = synth.even_partition(1000, 4)
    inp = synth.forward_inputs(16, 32, part, tau=0.7, seed=2, w_std=0.3)
    ids, y = synth.replay_ids(16, part, seed=3)
    a = oracle.top_p_replay(inp.X, inp.W, None, part, ids, y, inp.tau)
    rng = np.random.default_rng(0)
    ids2 = ids.copy()
    for t in range(16):
        live = ids2[t][ids2[t] != -1]
        free = 64 - live.size
        extra = rng.choice(live, size=min(free, 3))
        row = np.concatenate([live, extra, np.full(64 - live.size - extra.size, -1)])
        ids2[t] = rng.permutation(row)
    b = oracle.top_p_replay(inp.X, inp.W, None, part, ids2, y, inp.tau)
    np.testing.assert_array_equal(a.lse, b.lse)
    np.testing.assert_array_equal(a.logp, b.logp)


def test_replay_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.replay_set(np.array([3, 1000, -1]), 1000)
    with pytest.raises(ValueError):
        oracle.replay_set(np.array([-2]), 1000)


# --------------------------------------------------------------------- backward

def _loss(Xd, Wd, bd, ranges, Vr, y, tau, g):
    z = oracle.logits_f64(Xd, Wd, bd, ranges, Vr, tau)
    M = z.max(axis=1, keepdims=True)
    lse = (M + np.log(np.exp(z - M).sum(axis=1, keepdims=True)))[:, 0]
    return float(np.dot(g, z[np.arange(len(y)), y] - lse))


def test_backward_central_finite_differences():
    part = synth.ranges_partition(20, 24, [0, 10, 24])
    rng = np.random.default_rng(11)
    T, H, tau = 3, 5, 0.7
    Xd = rng.standard_normal((T, H))
    Wd = [rng.standard_normal((e - s, H)) * 0.5 for s, e in part.ranges]
    bd = [rng.standard_normal(e - s) * 0.5 for s, e in part.ranges]
    y = np.array([2, 19, 11])
    g = rng.standard_normal(T)
    r = oracle.backward_f64(Xd, Wd, bd, part.ranges, 20, y, tau, g)
    eps = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp = _loss(Xd, Wd, bd, part.ranges, 20, y, tau, g)
        arr[idx] = old - eps
        lm = _loss(Xd, Wd, bd, part.ranges, 20, y, tau, g)
        arr[idx] = old
        return (lp - lm) / (2 * eps)

    num_dX = np.array([[fd(Xd, (t, h)) for h in range(H)] for t in range(T)])
    np.testing.assert_allclose(r.dX, num_dX, rtol=1e-6, atol=1e-8)
    for k in range(2):
        Vk = Wd[k].shape[0]
        num_dW = np.array([[fd(Wd[k], (v, h)) for h in range(H)] for v in range(Vk)])
        num_db = np.array([fd(bd[k], (v,)) for v in range(Vk)])
        np.testing.assert_allclose(r.dW[k], num_dW, rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(r.db[k], num_db, rtol=1e-6, atol=1e-8)
    # padded ids (>= 20) have exactly zero gradient
    assert np.all(r.dW[1][10:] == 0) and np.all(r.db[1][10:] == 0)


def test_backward_bias_grad_sums_to_zero_per_row_invariant():
    part = synth.even_partition(300, 3)
    inp = synth.forward_inputs(7, 16, part, tau=0.7, seed=6, w_std=0.3, bias_std=0.1)
    g = synth.upstream_grad(7, seed=6)
    r = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    total = sum(float(d.sum()) for d in r.db)
    assert abs(total) < 1e-12


def test_backward_sampled_matches_full():
    part = synth.ranges_partition(200, 208, [0, 104, 208])
    inp = synth.forward_inputs(9, 16, part, tau=0.7, seed=8, w_std=0.3, bias_std=0.1)
    g = synth.upstream_grad(9, seed=8)
    full = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    dx_rows = [0, 4, 8]
    dw_rows = [[0, 50, 103], [0, 95, 96, 103]]       # 96.. are padded ids (>= 200)
    dX, dW, db = oracle.backward_sampled(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g,
                                         dx_rows, dw_rows)
    np.testing.assert_allclose(dX, full.dX[dx_rows], atol=1e-12)
    for k in range(2):
        np.testing.assert_allclose(dW[k], full.dW[k][dw_rows[k]], atol=1e-12)
        np.testing.assert_allclose(db[k], full.db[k][dw_rows[k]], atol=1e-12)


def test_backward_sampled_dx_only_matches_full():
    part = synth.ranges_partition(200, 208, [0, 104, 208])
    inp = synth.forward_inputs(9, 16, part, tau=0.7, seed=8, w_std=0.3, bias_std=0.1)
    g = synth.upstream_grad(9, seed=8)
    full = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    dX, dW, db = oracle.backward_sampled(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, [1, 7], [[], []])
    np.testing.assert_allclose(dX, full.dX[[1, 7]], atol=1e-12)
    assert dW[0].shape == (0, 16) and db[1].shape == (0,)



# ------------------------------------------------------- logits-gather replay

def _exact_logits_case(seed):
    """X, W with small-integer entries so that X W^T is exact in bf16: the unscaled
    logits a projection would produce can then be stored losslessly."""
    rng = np.random.default_rng(seed)
    part = synth.ranges_partition(50, 64, [0, 20, 20, 64])
    T, H = 6, 8
    Xf = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    Wf = rng.integers(-2, 3, size=(64, H)).astype(np.float32)
    X = synth.bf16_bits(Xf)
    W = [synth.bf16_bits(Wf[s:e]) for s, e in part.ranges]
    L = [synth.bf16_bits((Xf @ Wf[s:e].T).astype(np.float32)) for s, e in part.ranges]
    return part, X, W, L


def test_logits_gather_replay_equals_projection_replay_on_exact_logits():
    part, X, W, L = _exact_logits_case(0)
    ids, y = synth.replay_ids(6, part, seed=1, max_ids=30)
    a = oracle.top_p_replay(X, W, None, part, ids, y, 0.7)
    b = oracle.top_p_replay_from_logits(L, part, ids, y, 0.7)
    np.testing.assert_allclose(b.lse, a.lse, atol=1e-12)
    np.testing.assert_allclose(b.logp, a.logp, atol=1e-12)
    np.testing.assert_allclose(b.shard_lse, a.shard_lse, atol=1e-12)
    np.testing.assert_allclose(b.shard_t, a.shard_t, atol=1e-12)


def test_logits_gather_replay_whole_vocab_equals_logits_forward_and_brute_force():
    part = synth.ranges_partition(40, 48, [0, 16, 32, 48])
    L, y, tau = synth.logits_inputs(3, part, 0.7, seed=5, peak_frac=0.1)
    ids = np.full((3, 64), -1, np.int32)
    for t in range(3):
        ids[t, :40] = np.random.default_rng(t).permutation(40)
    r = oracle.top_p_replay_from_logits(L, part, ids, y, tau)
    f = oracle.forward_from_logits(L, part, y, tau)
    np.testing.assert_allclose(r.lse, f.lse, atol=1e-12)
    np.testing.assert_allclose(r.logp, f.logp, atol=1e-12)
    # brute force on row 0 over a 3-id set, temperature once
    ids1 = np.full((1, 64), -1, np.int32)
    ids1[0, :4] = [7, 33, 7, 20]
    r1 = oracle.top_p_replay_from_logits([x[:1] for x in L], part, ids1, np.array([33]), tau)
    zs = [_dec(L[0][0][7]) / tau, _dec(L[1][0][4]) / tau, _dec(L[2][0][1]) / tau]
    lse = math.log(math.fsum(math.exp(z) for z in zs))
    assert abs(r1.lse[0] - lse) < 1e-12 and abs(r1.logp[0] - (zs[2] - lse)) < 1e-12


# ------------------------------------------------------------ entropy gradient

def test_entropy_gradient_central_finite_differences():
    part = synth.ranges_partition(20, 24, [0, 10, 24])
    rng = np.random.default_rng(12)
    T, H, tau = 3, 5, 0.7
    Xd = rng.standard_normal((T, H))
    Wd = [rng.standard_normal((e - s, H)) * 0.5 for s, e in part.ranges]
    bd = [rng.standard_normal(e - s) * 0.5 for s, e in part.ranges]
    y = np.array([2, 19, 11])
    g = rng.standard_normal(T)
    hh = rng.standard_normal(T)
    r = oracle.backward_f64(Xd, Wd, bd, part.ranges, 20, y, tau, g, h=hh)

    def loss():
        z = oracle.logits_f64(Xd, Wd, bd, part.ranges, 20, tau)
        M = z.max(axis=1, keepdims=True)
        lse = (M + np.log(np.exp(z - M).sum(axis=1, keepdims=True)))[:, 0]
        p = np.exp(z - lse[:, None])
        ent = -(p * (z - lse[:, None])).sum(axis=1)
        return float(np.dot(g, z[np.arange(T), y] - lse) + np.dot(hh, ent))

    eps = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp_ = loss()
        arr[idx] = old - eps
        lm_ = loss()
        arr[idx] = old
        return (lp_ - lm_) / (2 * eps)

    np.testing.assert_allclose(r.dX, [[fd(Xd, (t, j)) for j in range(H)] for t in range(T)], rtol=1e-6, atol=1e-8)
    for k in range(2):
        Vk = Wd[k].shape[0]
        np.testing.assert_allclose(r.dW[k], [[fd(Wd[k], (v, j)) for j in range(H)] for v in range(Vk)],
                                   rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(r.db[k], [fd(bd[k], (v,)) for v in range(Vk)], rtol=1e-6, atol=1e-8)


def test_entropy_gradient_of_uniform_logits_vanishes():
    # z constant => p uniform, z - mu = 0: the entropy term adds nothing
    part = synth.even_partition(30, 1)
    X = np.zeros((2, 4), np.uint16)
    W = [np.zeros((30, 4), np.uint16)]
    g = np.array([0.5, -1.0])
    a = oracle.backward(X, W, None, part, np.array([1, 2]), 0.7, g)
    b = oracle.backward(X, W, None, part, np.array([1, 2]), 0.7, g, h=np.array([3.0, 7.0]))
    np.testing.assert_allclose(b.db[0], a.db[0], atol=1e-15)


# ------------------------------------------------------------ logits gradient

def _real_concat(L_bits, part):
    cols = []
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        if hi > vs:
            cols.append(oracle.bf16_to_f64(L_bits[k][:, : hi - vs]))
    return np.concatenate(cols, axis=1)


def test_logits_gradient_matches_torch_autograd_fp64():
    # independent library: torch's log_softmax and autograd in float64 on the CPU
    torch = pytest.importorskip("torch")
    part = synth.ranges_partition(90, 104, [0, 40, 40, 104])        # an empty shard, 14 padded ids
    T, tau = 6, 0.7
    L, y, _ = synth.logits_inputs(T, part, tau, seed=21)
    g = synth.upstream_grad(T, seed=21)
    h = synth.upstream_grad(T, seed=22)
    z = torch.tensor(_real_concat(L, part), dtype=torch.float64, requires_grad=True)
    ls = torch.log_softmax(z / tau, dim=1)
    logp = ls[torch.arange(T), torch.tensor(y, dtype=torch.long)]
    ent = -(ls.exp() * ls).sum(dim=1)
    loss = (torch.tensor(g, dtype=torch.float64) * logp).sum() + (torch.tensor(h, dtype=torch.float64) * ent).sum()
    loss.backward()
    ref = z.grad.numpy()
    dL = oracle.backward_from_logits(L, part, y, tau, g, h=h)
    assert [d.shape for d in dL] == [(T, 40), (T, 0), (T, 64)]
    np.testing.assert_allclose(np.concatenate([dL[0], dL[2][:, :50]], axis=1), ref, rtol=1e-10, atol=1e-13)
    assert np.all(dL[2][:, 50:] == 0)                                  # padded ids
    # logp term alone
    dL0 = oracle.backward_from_logits(L, part, y, tau, g)
    z.grad = None
    ls = torch.log_softmax(z / tau, dim=1)
    (torch.tensor(g, dtype=torch.float64) * ls[torch.arange(T), torch.tensor(y, dtype=torch.long)]).sum().backward()
    np.testing.assert_allclose(np.concatenate([dL0[0], dL0[2][:, :50]], axis=1), z.grad.numpy(), rtol=1e-10,
                               atol=1e-13)


def test_logits_gradient_rows_sum_to_zero_and_rows_select():
    part = synth.even_partition(500, 3, 510)
    T, tau = 9, 1.3
    L, y, _ = synth.logits_inputs(T, part, tau, seed=23)
    g = synth.upstream_grad(T, seed=23)
    h = synth.upstream_grad(T, seed=24)
    dL = oracle.backward_from_logits(L, part, y, tau, g, h=h)
    row_sum = sum(d.sum(axis=1) for d in dL)
    assert np.max(np.abs(row_sum)) < 1e-14
    rows = np.array([7, 2, 5])
    sub = oracle.backward_from_logits(L, part, y, tau, g, h=h, rows=rows)
    for a, b in zip(sub, dL):
        np.testing.assert_array_equal(a, b[rows])


def test_logits_gradient_chain_rule_to_projection_gradient():
    # With small-integer X and W the logits X W^T are integers, exact in bf16, so the
    # logits gradient must carry the projection gradient through L = X W^T:
    # dX = sum_k dL_k W_k, dW_k = dL_k^T X, db_k = sum_t dL_k.
    part = synth.ranges_partition(70, 80, [0, 30, 80])
    rng = np.random.default_rng(25)
    T, H, tau = 5, 6, 2.5
    Xi = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    Wi = [rng.integers(-2, 3, size=(e - s, H)).astype(np.float32) for s, e in part.ranges]
    X = synth.bf16_bits(Xi)
    W = [synth.bf16_bits(w) for w in Wi]
    L = [synth.bf16_bits(Xi @ w.T) for w in Wi]
    y = np.array([0, 69, 31, 29, 12])
    g = synth.upstream_grad(T, seed=25)
    h = synth.upstream_grad(T, seed=26)
    ref = oracle.backward(X, W, [np.zeros(e - s, np.uint16) for s, e in part.ranges], part, y, tau, g, h=h)
    dL = oracle.backward_from_logits(L, part, y, tau, g, h=h)
    dX = sum(d @ w.astype(np.float64) for d, w in zip(dL, Wi))
    np.testing.assert_allclose(dX, ref.dX, rtol=1e-12, atol=1e-14)
    for k in range(2):
        np.testing.assert_allclose(dL[k].T @ Xi.astype(np.float64), ref.dW[k], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dL[k].sum(axis=0), ref.db[k], rtol=1e-12, atol=1e-14)
