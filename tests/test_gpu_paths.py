"""GPU parity of the logits-reuse, compact top-p replay (and its dense keep-mask route)
and backward paths against the fp64 oracle, at sizes spanning several tiles with
ragged tails, padded ids and empty shards."""
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


# ----------------------------------------------------------------- logits reuse

def _strided_rows(a):
    """A [T, w] device view of bf16 bits `a` whose row stride is a multiple of 8 elements
    (16 bytes, as the library requires) with 8 elements to spare."""
    import torch
    T, w = a.shape
    ld = (w + 7) // 8 * 8 + 8
    buf = torch.zeros((T, ld), dtype=torch.bfloat16, device="cuda")
    buf[:, :w] = dev_bf16(a)
    return buf[:, :w]


@pytest.mark.parametrize("T,bounds,real", [
    (37, [0, 1000], 1000),
    (64, [0, 4099, 4099, 9000, 12301], 12290),     # ragged widths, empty shard, padding
    (5, [0, 7], 7),                                  # narrower than one vector
])
def test_logits_reuse_parity(lp, T, bounds, real):
    part = synth.ranges_partition(real, bounds[-1], bounds)
    L, y, tau = synth.logits_inputs(T, part, 0.7, seed=T)
    import torch
    # give every shard a padded row stride (multiple of 8) to exercise ld
    Ld = []
    for a in L:
        w = a.shape[1]
        if w == 0:
            Ld.append(None)
            continue
        ld = (w + 7) // 8 * 8 + 8
        buf = torch.zeros((T, ld), dtype=torch.bfloat16, device="cuda")
        buf[:, :w] = dev_bf16(a)
        Ld.append(buf[:, :w])
    out = lp.lp_forward_from_logits(Ld, part_of(part), dev_i32(y), tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward_from_logits(L, part, y, tau)
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"]), ref.entropy) <= TOL_ENT
    ss = _np(out["shard_stats"])
    for k, s in enumerate(ref.shards):
        assert max_abs(ss[k, 0], s.lse) <= TOL_LSE
        assert max_abs(ss[k, 1], s.t) <= TOL_LOGP
        assert max_abs(ss[k, 2], s.h) <= TOL_ENT


def test_logits_reuse_bitwise_and_batch_invariant(lp):
    import torch
    part = synth.even_partition(20000, 2)
    L, y, tau = synth.logits_inputs(96, part, 0.7, seed=3)
    Ld = [dev_bf16(a) for a in L]
    yd = dev_i32(y)
    a = lp.lp_forward_from_logits(Ld, part_of(part), yd, tau)
    b = lp.lp_forward_from_logits(Ld, part_of(part), yd, tau)
    c = lp.lp_forward_from_logits([x[40:].contiguous() for x in Ld], part_of(part), yd[40:].contiguous(), tau)
    for k in ("logp", "lse", "entropy"):
        assert torch.equal(a[k], b[k])
        assert torch.equal(a[k][40:], c[k])


@pytest.mark.parametrize("tau", [0.05, 0.7, 20.0])
def test_logits_reuse_masked_and_extreme_rows(lp, tau):
    """Rows built to stress the streaming fold: entries masked out with -inf (also a whole
    shard, and all but the target), large offsets, a far-below-the-rest half of the row, a
    single dominant logit, and rows whose maximum rises (or falls) with every element.
    A -inf logit and a finite one so low that exp underflows to exactly 0 in fp64 are the
    same to the definition, so the oracle sees -1e30 where the kernel sees -inf."""
    bounds, real = [0, 4101, 8203, 12000], 11990
    part = synth.ranges_partition(real, bounds[-1], bounds)
    T = 40
    tau = float(np.float32(tau))
    L, y, _ = synth.logits_inputs(T, part, tau, seed=17)
    full = np.concatenate(L, axis=1).view(np.uint16)
    x = (full.astype(np.uint32) << np.uint32(16)).view(np.float32).copy()
    rng = np.random.Generator(np.random.PCG64(99))
    y = y.astype(np.int64)
    mask = np.zeros(x.shape, bool)
    # row 0: 30 % of the real ids masked (never the target)
    mask[0, rng.choice(real, size=int(0.3 * real), replace=False)] = True
    # row 1: shard 1 masked entirely, target elsewhere
    mask[1, bounds[1]:bounds[2]] = True
    y[1] = 17
    # row 2: everything masked but the target
    mask[2, :real] = True
    y[2] = 9000
    mask[2, y[2]] = False
    mask[0, y[0]] = False
    # rows 3, 4: all logits shifted by +-300
    x[3] += 300.0
    x[4] -= 300.0
    # row 5: half of the ids at -1e30 (finite, far below every other logit)
    x[5, rng.choice(real, size=real // 2, replace=False)] = -1e30
    # row 6: one dominant logit
    x[6, 5000] = 200.0
    # rows 7, 8: maximum rising with every element / falling
    x[7, :real] = np.linspace(-50.0, 50.0, real)
    x[8, :real] = np.linspace(50.0, -50.0, real)
    bits = synth.bf16_bits(x.astype(np.float32))
    gpu_bits = bits.copy()
    gpu_bits[mask] = 0xFF80                        # bf16 -inf
    ora_bits = bits.copy()
    ora_bits[mask] = synth.bf16_bits(np.array([-1e30], np.float32))[0]
    split = lambda b: [np.ascontiguousarray(b[:, s:e]) for s, e in part.ranges]
    y32 = y.astype(np.int32)
    out = lp.lp_forward_from_logits([_strided_rows(a) for a in split(gpu_bits)], part_of(part), dev_i32(y32), tau,
                                    shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward_from_logits(split(ora_bits), part, y32, tau)
    lg, ls, en = _np(out["logp"]), _np(out["lse"]), _np(out["entropy"])
    assert np.all(np.isfinite(lg)) and np.all(np.isfinite(ls)) and np.all(np.isfinite(en))
    assert max_abs(lg, ref.logp) <= TOL_LOGP
    assert max_abs(ls, ref.lse) <= TOL_LSE
    assert max_abs(en, ref.entropy) <= TOL_ENT
    assert abs(lg[2]) <= 1e-5 and abs(en[2]) <= 1e-5   # one live id: p = 1
    ss = _np(out["shard_stats"])
    assert not np.isnan(ss).any()
    empty = np.stack([mask[:, s:min(e, real)].all(axis=1) for s, e in part.ranges])   # [K, T]
    assert empty[1, 1] and empty[0, 2] and empty[1, 2] and not empty[2, 2]
    for k in range(part.n_shards):
        live = ~empty[k]
        assert max_abs(ss[k, 0, live], ref.shards[k].lse[live]) <= TOL_LSE
        assert max_abs(ss[k, 2, live], ref.shards[k].h[live]) <= TOL_ENT
        # a shard whose ids are all masked is empty: LSE -inf, entropy 0
        assert np.all(np.isneginf(ss[k, 0, empty[k]])) and np.all(ss[k, 2, empty[k]] == 0.0)


# ----------------------------------------------------------------------- replay

def _mask_from_ids(ids, part):
    masks = [np.zeros((ids.shape[0], e - s), np.uint8) for s, e in part.ranges]
    for t in range(ids.shape[0]):
        for v in ids[t]:
            if v < 0:
                continue
            for k, (s, e) in enumerate(part.ranges):
                if s <= v < e:
                    masks[k][t, v - s] = 1
    return masks


@pytest.mark.parametrize("T,H,bounds,real,bias", [
    (200, 256, [0, 2500, 5000, 7500, 10000], 10000, None),
    (77, 136, [0, 3000, 3000, 8000, 8192], 8100, 0.2),     # empty shard, padding, H % 64 != 0
])
def test_replay_parity_and_dense_mask_bitwise(lp, T, H, bounds, real, bias):
    import torch
    part = synth.ranges_partition(real, bounds[-1], bounds)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=11, w_std=0.05, bias_std=bias)
    ids, y = synth.replay_ids(T, part, seed=12)
    X, W, b, _ = dev_inputs(inp)
    P = part_of(part)
    out = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids), dev_i32(y), inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, y, inp.tau)
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE
    ss = _np(out["shard_stats"])
    for k in range(part.n_shards):
        assert max_abs(ss[k, 0], ref.shard_lse[k]) <= TOL_LSE
        assert max_abs(ss[k, 1], ref.shard_t[k]) <= TOL_LOGP
    # the dense keep-mask route gives the same bits
    masks = [dev_i32(m).to(torch.uint8) if m.shape[1] else None for m in _mask_from_ids(ids, part)]
    dm = lp.lp_top_p_replay_dense_mask(X, W, b, P, masks, dev_i32(y), inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    for k in ("logp", "lse", "shard_stats"):
        assert torch.equal(dm[k], out[k]), k
    # slot order and duplicates do not change a bit
    rng = np.random.default_rng(0)
    ids2 = ids.copy()
    for t in range(T):
        live = ids2[t][ids2[t] >= 0]
        extra = rng.choice(live, size=min(3, 64 - live.size))
        row = np.concatenate([live, extra, np.full(64 - live.size - extra.size, -1)])
        ids2[t] = rng.permutation(row)
    o2 = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids2), dev_i32(y), inp.tau, shard_stats=True)
    for k in ("logp", "lse", "shard_stats"):
        assert torch.equal(o2[k], out[k]), k
    # batch invariance
    o3 = lp.lp_top_p_replay(X[10:].contiguous(), W, b, P, dev_i32(ids[10:]), dev_i32(y[10:]), inp.tau)
    assert torch.equal(o3["logp"], out["logp"][10:]) and torch.equal(o3["lse"], out["lse"][10:])


def test_replay_adversarial_slot_patterns(lp):
    """Slot patterns that stress the in-warp sort and deduplication: 64 distinct ids in
    descending and in ascending order, one id 64 times, the two ends of the vocabulary,
    ids alternating between the first and last shard, one id among 63 empty slots (first
    or last slot), and pairs of equal ids at every other slot."""
    import torch
    bounds, real = [0, 1000, 2000, 3000, 4096], 4090
    part = synth.ranges_partition(real, bounds[-1], bounds)
    T, H = 10, 128
    inp = synth.forward_inputs(T, H, part, tau=0.6, seed=31, w_std=0.2, bias_std=0.1)
    ids = np.full((T, 64), -1, np.int32)
    ids[0] = np.arange(4000, 3936, -1)
    ids[1] = np.arange(100, 164)
    ids[2] = 777
    ids[3, :2] = [0, real - 1]
    ids[4] = np.where(np.arange(64) % 2 == 0, np.arange(64) * 7, real - 1 - np.arange(64) * 5)
    ids[5, 0] = 2500
    ids[6, 63] = 2500
    ids[7] = np.repeat(np.arange(3000, 3032), 2)
    ids[8, ::2] = np.arange(32) * 100
    ids[9] = np.random.default_rng(5).permutation(np.arange(1990, 2054))
    y = np.array([3937, 163, 777, real - 1, 0, 2500, 2500, 3031, 3150, 2000], np.int32)
    X, W, b, _ = dev_inputs(inp)
    P = part_of(part)
    out = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids), dev_i32(y), inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, y, inp.tau)
    lg, ls = _np(out["logp"]), _np(out["lse"])
    fin = np.isfinite(ref.logp)
    assert np.array_equal(np.isfinite(lg), fin) and np.array_equal(np.isfinite(ls), np.isfinite(ref.lse))
    assert max_abs(lg[fin], ref.logp[fin]) <= TOL_LOGP
    assert max_abs(ls, ref.lse) <= TOL_LSE
    assert not fin[8] and np.all(fin[[0, 1, 2, 3, 4, 5, 6, 7, 9]])   # row 8: target not in its set
    assert abs(lg[2]) <= 1e-5 and abs(lg[5]) <= 1e-5                  # a single id: p = 1
    ss = _np(out["shard_stats"])
    for k in range(part.n_shards):
        assert max_abs(ss[k, 0], ref.shard_lse[k]) <= TOL_LSE
        assert max_abs(ss[k, 1], ref.shard_t[k]) <= TOL_LOGP
    # the same rows with their slots reversed give the same bits
    rev = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids[:, ::-1].copy()), dev_i32(y), inp.tau, shard_stats=True)
    for key in ("logp", "lse", "shard_stats"):
        assert torch.equal(rev[key], out[key]), key


def test_replay_whole_vocab_matches_dense_forward(lp):
    part = synth.ranges_partition(60, 64, [0, 16, 32, 48, 64])
    inp = synth.forward_inputs(9, 64, part, tau=0.7, seed=4, w_std=0.3, bias_std=0.2)
    ids = np.full((9, 64), -1, np.int32)
    for t in range(9):
        ids[t, :60] = np.random.default_rng(t).permutation(60)
    X, W, b, y = dev_inputs(inp)
    rep = lp.lp_top_p_replay(X, W, b, part_of(part), dev_i32(ids), y, inp.tau)
    fwd = lp.lp_forward(X, W, b, part_of(part), y, inp.tau)
    assert max_abs(_np(rep["lse"]), _np(fwd["lse"])) <= TOL_LSE
    assert max_abs(_np(rep["logp"]), _np(fwd["logp"])) <= TOL_LOGP


def test_replay_errors_and_empty_rows(lp):
    part = synth.even_partition(1000, 2)
    inp = synth.forward_inputs(4, 64, part, tau=0.7, seed=9)
    X, W, b, _ = dev_inputs(inp)
    ids = np.full((4, 64), -1, np.int32)
    ids[0, :3] = [5, 600, 5]
    ids[1, 0] = 1000                     # out of range: device error, row fails closed
    # row 2: no ids at all; row 3: target not in the set
    ids[3, :2] = [7, 8]
    y = np.array([600, 3, 4, 9], np.int32)
    out = lp.lp_top_p_replay(X, W, b, part_of(part), dev_i32(ids), dev_i32(y), inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 6
    lg, ls = _np(out["logp"]), _np(out["lse"])
    assert np.isfinite(lg[0]) and np.isfinite(ls[0])
    assert np.isneginf(lg[1]) and np.isneginf(ls[1])
    assert np.isneginf(lg[2]) and np.isneginf(ls[2])
    assert np.isneginf(lg[3]) and np.isfinite(ls[3])
    ss = _np(out["shard_stats"])
    assert not np.any(np.isnan(ss))
    assert np.isneginf(ss[1, 0, 3]) and ss[1, 1, 3] == 0.0      # row 3 has no id in shard 1


# --------------------------------------------------------------------- backward

def test_minus_inf_bias_masks_ids_forward_and_backward(lp):
    """A bias of -inf masks an id out of the softmax (p = 0): forward statistics and every
    gradient stay finite, and masked ids get exactly zero dW and db. As in the logits-reuse
    test, the oracle sees -1e30, whose exponential is exactly 0 in fp64 as well. Masked: a
    whole 256-id vocabulary block and 15 % of the other ids (never a target)."""
    import torch
    bounds, real = [0, 600, 1200], 1190
    part = synth.ranges_partition(real, bounds[-1], bounds)
    T, H = 70, 96
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=61, w_std=0.1, bias_std=0.2)
    rng = np.random.default_rng(62)
    masked = np.zeros(bounds[-1], bool)
    masked[256:512] = True
    masked[rng.choice(real, size=int(0.15 * real), replace=False)] = True
    masked[real:] = False
    live = np.flatnonzero(~masked[:real])
    y = rng.choice(live, size=T).astype(np.int32)
    neg_inf = np.uint16(0xFF80)
    very_low = synth.bf16_bits(np.array([-1e30], np.float32))[0]
    b_gpu, b_ora = [], []
    for (s, e), bk in zip(part.ranges, inp.bias):
        m = masked[s:e]
        b_gpu.append(np.where(m, neg_inf, bk).astype(np.uint16))
        b_ora.append(np.where(m, very_low, bk).astype(np.uint16))
    X, W, _, _ = dev_inputs(inp)
    b = [dev_bf16(x) for x in b_gpu]
    P = part_of(part)
    yd = dev_i32(y)
    fwd = lp.lp_forward(X, W, b, P, yd, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward(inp.X, inp.W, b_ora, part, y, inp.tau)
    lg, ls, en = _np(fwd["logp"]), _np(fwd["lse"]), _np(fwd["entropy"])
    assert np.all(np.isfinite(lg)) and np.all(np.isfinite(ls)) and np.all(np.isfinite(en))
    assert max_abs(lg, ref.logp) <= TOL_LOGP
    assert max_abs(ls, ref.lse) <= TOL_LSE
    assert max_abs(en, ref.entropy) <= TOL_ENT
    assert not np.isnan(_np(fwd["shard_stats"])).any()
    g = synth.upstream_grad(T, seed=63)
    h = synth.upstream_grad(T, seed=64)
    bw = lp.lp_backward(X, W, b, P, yd, inp.tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                        grad_entropy=dev_f32(h))
    assert lp.lp_get_device_error() == 0
    bref = oracle.backward(inp.X, inp.W, b_ora, part, y, inp.tau, g, h=h)
    assert rel_fro(_np(bw["dX"]), bref.dX) <= TOL_GRAD_REL
    for k, (s, e) in enumerate(part.ranges):
        dw, db = _np(bw["dW"][k]), _np(bw["db"][k])
        assert np.all(np.isfinite(dw)) and np.all(np.isfinite(db))
        assert rel_fro(dw, bref.dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(db, bref.db[k]) <= TOL_GRAD_REL, k
        m = masked[s:e]
        assert np.all(dw[m] == 0) and np.all(db[m] == 0), k



@pytest.mark.parametrize("T,H,bounds,real,bias", [
    (64, 256, [0, 1000], 1000, None),
    (200, 192, [0, 700, 700, 1500, 2048], 2000, 0.3),    # empty shard, padding, ragged rows
    (130, 520, [0, 300, 640], 600, 0.1),                 # H % 256 != 0, shard widths not multiples of 64
])
def test_backward_parity(lp, T, H, bounds, real, bias):
    part = synth.ranges_partition(real, bounds[-1], bounds)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=T, w_std=0.05, bias_std=bias)
    g = synth.upstream_grad(T, seed=T)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    assert rel_fro(_np(bw["dX"]), ref.dX) <= TOL_GRAD_REL
    for k, (s, e) in enumerate(part.ranges):
        if e == s:
            continue
        assert rel_fro(_np(bw["dW"][k]), ref.dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(_np(bw["db"][k]), ref.db[k]) <= TOL_GRAD_REL, k
        # padded ids get exactly zero gradient
        pad = slice(max(0, real - s), e - s)
        assert np.all(_np(bw["dW"][k])[pad] == 0) and np.all(_np(bw["db"][k])[pad] == 0)


def test_backward_bitwise_repeatable_and_dx_batch_invariant(lp):
    import torch
    part = synth.ranges_partition(3000, 3072, [0, 1500, 3072])
    inp = synth.forward_inputs(300, 256, part, tau=0.7, seed=2, bias_std=0.1)
    g = dev_f32(synth.upstream_grad(300, seed=2))
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    a = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], g)
    c = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], g)
    assert torch.equal(a["dX"], c["dX"])
    for k in range(2):
        assert torch.equal(a["dW"][k], c["dW"][k]) and torch.equal(a["db"][k], c["db"][k])
    # a row's dX depends only on that row: the same rows in another batch give the same bits,
    # also with 70000 K columns split into two fixed K ranges
    for lo, hi in ((0, 1), (37, 300), (129, 257)):
        sub = lp.lp_backward(X[lo:hi].contiguous(), W, b, P, y[lo:hi].contiguous(), inp.tau,
                             fwd["lse"][lo:hi].contiguous(), g[lo:hi].contiguous())
        assert torch.equal(sub["dX"], a["dX"][lo:hi]), (lo, hi)
    part2 = synth.ranges_partition(70000, 70016, [0, 35008, 70016])
    inp2 = synth.forward_inputs(260, 128, part2, tau=0.7, seed=3, w_std=0.05)
    X2, W2, _, y2 = dev_inputs(inp2)
    P2 = part_of(part2)
    g2 = dev_f32(synth.upstream_grad(260, seed=3))
    f2 = lp.lp_forward(X2, W2, None, P2, y2, inp2.tau)
    full = lp.lp_backward(X2, W2, None, P2, y2, inp2.tau, f2["lse"], g2)["dX"]
    sub = lp.lp_backward(X2[3:200].contiguous(), W2, None, P2, y2[3:200].contiguous(), inp2.tau,
                         f2["lse"][3:200].contiguous(), g2[3:200].contiguous())["dX"]
    assert torch.equal(sub, full[3:200])


# ---------------------------------------------------------- logits-gather replay

@pytest.mark.parametrize("T,bounds,real", [
    (150, [0, 2500, 5000, 7500, 10000], 10000),
    (33, [0, 3000, 3000, 8000, 8192], 8100),          # empty shard, padded ids
])
def test_replay_from_logits_parity(lp, T, bounds, real):
    import torch
    part = synth.ranges_partition(real, bounds[-1], bounds)
    L, _, tau = synth.logits_inputs(T, part, 0.7, seed=T)
    ids, y = synth.replay_ids(T, part, seed=T + 1)
    Ld = [dev_bf16(a) if a.shape[1] else None for a in L]
    out = lp.lp_top_p_replay_from_logits(Ld, part_of(part), dev_i32(ids), dev_i32(y), tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    ref = oracle.top_p_replay_from_logits(L, part, ids, y, tau)
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE
    ss = _np(out["shard_stats"])
    for k in range(part.n_shards):
        assert max_abs(ss[k, 0], ref.shard_lse[k]) <= TOL_LSE
        assert max_abs(ss[k, 1], ref.shard_t[k]) <= TOL_LOGP
    again = lp.lp_top_p_replay_from_logits(Ld, part_of(part), dev_i32(ids), dev_i32(y), tau, shard_stats=True)
    for k in ("logp", "lse", "shard_stats"):
        assert torch.equal(again[k], out[k])


def test_replay_from_exact_logits_is_bitwise_the_projection_replay(lp):
    # small-integer X and W: every fp32 dot product is exact and equals the bf16 logit,
    # so scoring from logits and from x . W give the same bits
    import torch
    rng = np.random.default_rng(3)
    part = synth.ranges_partition(500, 512, [0, 200, 200, 512])
    T, H = 40, 32
    Xf = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    Wf = rng.integers(-2, 3, size=(512, H)).astype(np.float32)
    X = dev_bf16(synth.bf16_bits(Xf))
    W = [dev_bf16(synth.bf16_bits(Wf[s:e])) if e > s else None for s, e in part.ranges]
    L = [dev_bf16(synth.bf16_bits((Xf @ Wf[s:e].T).astype(np.float32))) if e > s else None for s, e in part.ranges]
    ids, y = synth.replay_ids(T, part, seed=4)
    P = part_of(part)
    a = lp.lp_top_p_replay(X, W, None, P, dev_i32(ids), dev_i32(y), 0.7, shard_stats=True)
    b = lp.lp_top_p_replay_from_logits(L, P, dev_i32(ids), dev_i32(y), 0.7, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    for k in ("logp", "lse", "shard_stats"):
        assert torch.equal(a[k], b[k]), k


# ------------------------------------------------------------ entropy gradient

@pytest.mark.parametrize("T,H,bounds,real,bias", [
    (96, 256, [0, 1000], 1000, None),
    (150, 192, [0, 700, 700, 1500, 2048], 2000, 0.3),
])
def test_backward_with_entropy_gradient_parity(lp, T, H, bounds, real, bias):
    part = synth.ranges_partition(real, bounds[-1], bounds)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=T + 1, w_std=0.05, bias_std=bias)
    g = synth.upstream_grad(T, seed=T)
    h = synth.upstream_grad(T, seed=T + 100)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                        grad_entropy=dev_f32(h))
    assert lp.lp_get_device_error() == 0
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, h=h)
    assert rel_fro(_np(bw["dX"]), ref.dX) <= TOL_GRAD_REL
    for k, (s, e) in enumerate(part.ranges):
        if e == s:
            continue
        assert rel_fro(_np(bw["dW"][k]), ref.dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(_np(bw["db"][k]), ref.db[k]) <= TOL_GRAD_REL, k
    # and the entropy term is really there: without it the result is far off
    plain = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    assert rel_fro(plain.dX, ref.dX) > 3 * TOL_GRAD_REL


def test_many_row_blocks_forward_replay_logits_backward(lp):
    # T = 70000 rows (547 row blocks, 8750 replay CTAs) with a small vocabulary: sampled rows
    # against the oracle, and dW / db in full (the oracle's T x V x H is small here)
    import torch
    part = synth.ranges_partition(1000, 1024, [0, 512, 1024])
    T, H = 70000, 64
    inp = synth.forward_inputs(T, H, part, tau=0.8, seed=77, w_std=0.3, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, T - 129, T - 1],
                                     np.random.default_rng(78).choice(T, 200, replace=False)]))
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, rows=rows)
    assert max_abs(_np(fwd["logp"])[rows], ref.logp) <= TOL_LOGP
    assert max_abs(_np(fwd["entropy"])[rows], ref.entropy) <= TOL_ENT
    ids, yr = synth.replay_ids(T, part, seed=79)
    rp = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids), dev_i32(yr), inp.tau)
    rref = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, yr, inp.tau, rows=rows)
    assert max_abs(_np(rp["lse"])[rows], rref.lse) <= TOL_LSE
    g = synth.upstream_grad(T, seed=80)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0
    bref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    assert rel_fro(_np(bw["dX"])[rows], bref.dX[rows]) <= TOL_GRAD_REL
    for k in range(2):
        assert rel_fro(_np(bw["dW"][k]), bref.dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(_np(bw["db"][k]), bref.db[k]) <= TOL_GRAD_REL, k
    # the first 4096 rows alone give the same forward bits (batch invariance at this size)
    head = lp.lp_forward(X[:4096].contiguous(), W, b, P, y[:4096].contiguous(), inp.tau)
    assert torch.equal(head["logp"], fwd["logp"][:4096]) and torch.equal(head["lse"], fwd["lse"][:4096])
    # the logits-reuse route over the same 70000 rows (one CTA per row)
    L, yl, tau = synth.logits_inputs(T, part, 0.8, seed=81)
    lf = lp.lp_forward_from_logits([dev_bf16(a) for a in L], P, dev_i32(yl), tau)
    assert lp.lp_get_device_error() == 0
    lref = oracle.forward_from_logits(L, part, yl, tau, rows=rows)
    assert max_abs(_np(lf["logp"])[rows], lref.logp) <= TOL_LOGP
    assert max_abs(_np(lf["entropy"])[rows], lref.entropy) <= TOL_ENT


def test_projection_row_chunks_forward_and_backward(lp):
    # T = 9000 rows at H = 4096 makes the projection GEMMs take their rows in three chunks
    # (4096, 4096, 808): the forward and dX must equal the same rows computed as their own
    # batches bit for bit, and dW / db must match the oracle over all 9000 rows
    import torch
    part = synth.ranges_partition(4000, 4096, [0, 2048, 4096])
    T, H = 9000, 4096
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=90, w_std=0.01, bias_std=0.05)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    g = dev_f32(synth.upstream_grad(T, seed=91))
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], g)
    assert lp.lp_get_device_error() == 0
    for lo, hi in ((0, 4096), (4096, 8192), (8192, 9000), (3000, 5000)):
        sub = lp.lp_forward(X[lo:hi].contiguous(), W, b, P, y[lo:hi].contiguous(), inp.tau)
        assert torch.equal(sub["logp"], fwd["logp"][lo:hi]) and torch.equal(sub["lse"], fwd["lse"][lo:hi]), (lo, hi)
        sb = lp.lp_backward(X[lo:hi].contiguous(), W, b, P, y[lo:hi].contiguous(), inp.tau,
                            fwd["lse"][lo:hi].contiguous(), g[lo:hi].contiguous())
        assert torch.equal(sb["dX"], bw["dX"][lo:hi]), (lo, hi)
    rows = np.unique(np.concatenate([[0, 4095, 4096, 8191, 8192, 8999],
                                     np.random.default_rng(92).choice(T, 40, replace=False)]))
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, rows=rows)
    assert max_abs(_np(fwd["logp"])[rows], ref.logp) <= TOL_LOGP
    bref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, _np(g))
    assert rel_fro(_np(bw["dX"])[rows], bref.dX[rows]) <= TOL_GRAD_REL
    for k in range(2):
        assert rel_fro(_np(bw["dW"][k]), bref.dW[k]) <= TOL_GRAD_REL, k
        assert rel_fro(_np(bw["db"][k]), bref.db[k]) <= TOL_GRAD_REL, k
