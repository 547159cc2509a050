"""Seeded random sweep: small configurations drawn at random (rows, hidden size, shard
layout with empty and all-padding shards, bias on/off, temperature), and a few fixed tiny
shapes, through every entry point, each compared with the fp64 oracle; the option and host entry points are checked
bit for bit against their plain counterparts on the same configurations."""
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


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.integers(1, 400))
    H = int(rng.choice([8, 16, 64, 72, 136, 256, 520]))
    n = int(rng.integers(1, 6))
    vpad = int(rng.integers(n * 8, 3000)) // 8 * 8
    cuts = np.sort(rng.choice(np.arange(0, vpad + 1, 8), size=n - 1, replace=True))   # empty shards allowed
    bounds = [0] + [int(c) for c in cuts] + [vpad]
    vreal = int(rng.integers(1, vpad + 1))
    bias = None if rng.random() < 0.5 else float(rng.choice([0.05, 0.5]))
    tau = float(rng.choice([0.3, 0.7, 1.0, 2.5]))
    return T, H, bounds, vreal, vpad, bias, tau


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration_all_entry_points(lp, seed):
    _check_all_entry_points(lp, *_random_case(seed), seed=seed)


# a few rows, H = 16 or 8, vocabularies smaller than one 256-id tile: shards of 8 ids, an
# empty shard, padding inside the only tile
@pytest.mark.parametrize("T,H,bounds,vreal,bias,tau", [
    (1, 16, [0, 40, 96], 90, 0.5, 0.7),
    (2, 16, [0, 0, 200], 200, None, 1.0),
    (3, 16, [0, 8, 16, 24], 20, 0.05, 2.5),
    (3, 8, [0, 248], 247, None, 0.3),
])
def test_tiny_shapes_all_entry_points(lp, T, H, bounds, vreal, bias, tau):
    _check_all_entry_points(lp, T, H, bounds, vreal, bounds[-1], bias, tau, seed=100 * T + H)


def test_most_shards_all_entry_points(lp):
    """LP_MAX_SHARDS = 8 shards (every per-shard slot in use, the last tensor map included):
    an empty shard, two 8-id shards, widths that are not multiples of the 256-id tile, padding
    in the last shard."""
    bounds = [0, 512, 520, 1000, 1000, 1600, 2048, 2056, 2600]
    assert len(bounds) - 1 == 8
    _check_all_entry_points(lp, 300, 136, bounds, 2590, 2600, 0.05, 0.7, seed=8)


def _check_all_entry_points(lp, T, H, bounds, vreal, vpad, bias, tau, seed):
    import torch
    part = synth.ranges_partition(vreal, vpad, bounds)
    inp = synth.forward_inputs(T, H, part, tau=tau, seed=seed, w_std=0.5 / np.sqrt(H), bias_std=bias)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    ctx = f"T={T} H={H} bounds={bounds} real={vreal} bias={bias} tau={tau}"

    fwd = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0, ctx
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    assert max_abs(_np(fwd["logp"]), ref.logp) <= TOL_LOGP, ctx
    assert max_abs(_np(fwd["lse"]), ref.lse) <= TOL_LSE, ctx
    assert max_abs(_np(fwd["entropy"]), ref.entropy) <= TOL_ENT, ctx
    ss = _np(fwd["shard_stats"])
    for k, s in enumerate(ref.shards):
        assert max_abs(ss[k, 0], s.lse) <= TOL_LSE, ctx
        assert max_abs(ss[k, 1], s.t) <= TOL_LOGP, ctx

    # the same logits, materialised and reused (unscaled, row stride padded to 8)
    z = oracle.logits_from_bits(inp.X, inp.W, inp.bias, part, 1.0)       # X W^T + b, real ids
    Lbits = []
    for k, (s, e) in enumerate(part.ranges):
        w = e - s
        full = np.zeros((T, w), np.float32)
        hi = min(e, vreal)
        if hi > s:
            full[:, :hi - s] = z[:, s:hi]
        Lbits.append(synth.bf16_bits(full))
    Ld = []
    for a in Lbits:
        w = a.shape[1]
        if w == 0:
            Ld.append(None)
            continue
        buf = torch.zeros((T, (w + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")
        buf[:, :w] = dev_bf16(a)
        Ld.append(buf[:, :w])
    lg = lp.lp_forward_from_logits(Ld, P, y, inp.tau)
    lref = oracle.forward_from_logits(Lbits, part, inp.y, inp.tau)
    assert lp.lp_get_device_error() == 0, ctx
    assert max_abs(_np(lg["lse"]), lref.lse) <= TOL_LSE, ctx
    assert max_abs(_np(lg["entropy"]), lref.entropy) <= TOL_ENT, ctx

    # replay, both score sources
    ids, yr = synth.replay_ids(T, part, seed=seed)
    rp = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids), dev_i32(yr), inp.tau)
    rref = oracle.top_p_replay(inp.X, inp.W, inp.bias, part, ids, yr, inp.tau)
    assert lp.lp_get_device_error() == 0, ctx
    assert max_abs(_np(rp["lse"]), rref.lse) <= TOL_LSE, ctx
    assert max_abs(_np(rp["logp"]), rref.logp) <= TOL_LOGP, ctx
    # the dense keep-mask route over the same sets: bitwise equal, whatever the shard
    # offsets and empty shards of this partition
    ids_d = dev_i32(ids)
    masks = []
    for k, (s0, e0) in enumerate(part.ranges):
        if e0 == s0:
            masks.append(None)
            continue
        m = torch.zeros((T, e0 - s0), dtype=torch.uint8, device="cuda")
        sel = (ids_d >= s0) & (ids_d < e0)
        rr = torch.arange(T, device="cuda").unsqueeze(1).expand_as(ids_d)[sel]
        m[rr.long(), (ids_d[sel] - s0).long()] = 1
        masks.append(m)
    dm = lp.lp_top_p_replay_dense_mask(X, W, b, P, masks, dev_i32(yr), inp.tau)
    assert torch.equal(dm["lse"], rp["lse"]) and torch.equal(dm["logp"], rp["logp"]), ctx
    rq = lp.lp_top_p_replay_from_logits(Ld, P, dev_i32(ids), dev_i32(yr), inp.tau)
    qref = oracle.top_p_replay_from_logits(Lbits, part, ids, yr, inp.tau)
    assert max_abs(_np(rq["lse"]), qref.lse) <= TOL_LSE, ctx

    # backward of logp alone (the G epilogue without an entropy gradient)
    g = synth.upstream_grad(T, seed=seed)
    bw0 = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g))
    assert lp.lp_get_device_error() == 0, ctx
    bref0 = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
    assert rel_fro(_np(bw0["dX"]), bref0.dX) <= TOL_GRAD_REL, ctx
    for k, (s, e) in enumerate(part.ranges):
        if e == s:
            continue
        assert rel_fro(_np(bw0["dW"][k]), bref0.dW[k]) <= TOL_GRAD_REL, (ctx, k)
        assert rel_fro(_np(bw0["db"][k]), bref0.db[k]) <= TOL_GRAD_REL, (ctx, k)

    # backward with the entropy term
    h = synth.upstream_grad(T, seed=seed + 50)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                        grad_entropy=dev_f32(h))
    assert lp.lp_get_device_error() == 0, ctx
    bref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g, h=h)
    assert rel_fro(_np(bw["dX"]), bref.dX) <= TOL_GRAD_REL, ctx
    for k, (s, e) in enumerate(part.ranges):
        if e == s:
            continue
        assert rel_fro(_np(bw["dW"][k]), bref.dW[k]) <= TOL_GRAD_REL, (ctx, k)
        assert rel_fro(_np(bw["db"][k]), bref.db[k]) <= TOL_GRAD_REL, (ctx, k)

    # the same gradient with a bf16 dX, and accumulated onto random fp32 buffers
    dX16 = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                             grad_entropy=dev_f32(h), dx_dtype=torch.bfloat16)["dX"]
    assert torch.equal(dX16, bw["dX"].to(torch.bfloat16)), ctx
    gen = torch.Generator(device="cuda").manual_seed(seed)
    dW0 = [None if d is None else torch.randn(d.shape, generator=gen, device="cuda") for d in bw["dW"]]
    db0 = [None if d is None else torch.randn(d.shape, generator=gen, device="cuda") for d in bw["db"]]
    acc = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                            grad_entropy=dev_f32(h), accumulate=True,
                            dW=[None if d is None else d.clone() for d in dW0],
                            db=[None if d is None else d.clone() for d in db0])
    for k, (s0, e0) in enumerate(part.ranges):
        if e0 == s0:
            continue
        r = max(min(e0, vreal) - s0, 0)
        assert torch.equal(acc["dW"][k][:r], dW0[k][:r] + bw["dW"][k][:r]), (ctx, k)
        assert torch.equal(acc["dW"][k][r:], dW0[k][r:]), (ctx, k)
        assert torch.equal(acc["db"][k][:r], db0[k][:r] + bw["db"][k][:r]), (ctx, k)

    # gradient with respect to the reused logits, against the oracle
    dL = lp.lp_backward_from_logits(Ld, P, y, inp.tau, lg["lse"], dev_f32(g), entropy=lg["entropy"],
                                    grad_entropy=dev_f32(h), out_dtype=torch.float32)
    dref = oracle.backward_from_logits(Lbits, part, inp.y, inp.tau, g, h=h)
    for k, (d, r) in enumerate(zip(dL, dref)):
        if r.shape[1] == 0:
            assert d is None, (ctx, k)
            continue
        assert rel_fro(_np(d), r) <= TOL_GRAD_REL, (ctx, k)

    # the host entry point gives the device forward's bits
    hX = torch.from_numpy(inp.X.view(np.int16)).view(torch.bfloat16)
    ho = lp.lp_forward_host(hX, W, b, P, torch.from_numpy(inp.y), inp.tau, shard_stats=True)
    for k in ("logp", "lse", "entropy", "shard_stats"):
        assert torch.equal(ho[k], fwd[k].cpu()), (ctx, k)
    assert lp.lp_get_device_error() == 0, ctx
