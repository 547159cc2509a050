"""Fail-closed behaviour of every entry point on bad data found on the device: the
sticky error word reports it, the affected rows get logp = -inf (replay: LSE -inf too),
nothing turns into NaN, and rows without a valid target or a finite LSE get no gradient."""
import numpy as np
import pytest

import oracle
import synth
from lp_util import TOL_GRAD_REL, dev_bf16, dev_f32, dev_i32, dev_inputs, part_of, rel_fro

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


def test_logits_reuse_target_out_of_range(lp):
    part = synth.even_partition(2000, 2)
    L, y, tau = synth.logits_inputs(6, part, 0.7, seed=1)
    y[2] = 2000
    out = lp.lp_forward_from_logits([dev_bf16(a) for a in L], part_of(part), dev_i32(y), tau)
    assert lp.lp_get_device_error() == 5
    lg = _np(out["logp"])
    assert np.isneginf(lg[2]) and np.all(np.isfinite(np.delete(lg, 2)))
    assert not np.isnan(_np(out["lse"])).any() and not np.isnan(_np(out["entropy"])).any()


def test_logits_gather_replay_bad_id_and_target(lp):
    part = synth.even_partition(2000, 2)
    L, _, tau = synth.logits_inputs(4, part, 0.7, seed=2)
    ids = np.full((4, 64), -1, np.int32)
    ids[0, :2] = [5, 1500]
    ids[1, :2] = [5, 4000]                  # out of range id
    ids[2, :1] = [7]
    ids[3, :1] = [9]
    y = np.array([1500, 5, -3, 9], np.int32)  # row 2: invalid target
    out = lp.lp_top_p_replay_from_logits([dev_bf16(a) for a in L], part_of(part), dev_i32(ids), dev_i32(y), tau)
    err = lp.lp_get_device_error()
    assert err in (5, 6)                     # the first error recorded wins
    lg, ls = _np(out["logp"]), _np(out["lse"])
    assert np.isfinite(lg[0]) and np.isneginf(lg[1]) and np.isneginf(ls[1])
    assert np.isneginf(lg[2]) and np.isfinite(ls[2])
    assert lg[3] == 0.0 or abs(lg[3]) < 1e-6


def test_dense_mask_with_more_than_64_ids_is_an_error(lp):
    import torch
    part = synth.even_partition(1000, 1)
    inp = synth.forward_inputs(3, 64, part, tau=0.7, seed=3)
    X, W, _, _ = dev_inputs(inp)
    mask = torch.zeros((3, 1000), dtype=torch.uint8, device="cuda")
    mask[0, :10] = 1
    mask[1, :65] = 1                         # 65 kept ids
    mask[2, 500] = 1
    y = dev_i32(np.array([3, 3, 500], np.int32))
    out = lp.lp_top_p_replay_dense_mask(X, W, None, part_of(part), [mask], y, inp.tau)
    assert lp.lp_get_device_error() == 9      # LP_ERR_REPLAY_TOO_MANY_IDS
    lse, lg = _np(out["lse"]), _np(out["logp"])
    assert np.isfinite(lse[0]) and np.isfinite(lse[2])
    assert np.isneginf(lse[1]) and np.isneginf(lg[1])     # the overfull row fails closed


def test_backward_rows_without_target_or_lse_get_no_gradient(lp):
    import torch
    part = synth.ranges_partition(900, 1024, [0, 512, 1024])
    inp = synth.forward_inputs(40, 64, part, tau=0.7, seed=4, w_std=0.1, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    g = synth.upstream_grad(40, seed=4)
    lse = fwd["lse"].clone()
    lse[7] = float("-inf")                   # e.g. a row whose forward failed closed
    g[11] = float("nan")                     # a non-finite upstream gradient
    yb = y.clone()
    yb[13] = 950                             # a padded id: invalid target
    bw = lp.lp_backward(X, W, b, P, yb, inp.tau, lse, dev_f32(g))
    assert lp.lp_get_device_error() == 0
    dX = _np(bw["dX"])
    assert np.all(dX[[7, 11, 13]] == 0) and np.isfinite(dX).all()
    # the other rows match the oracle restricted to them
    keep = np.array([r for r in range(40) if r not in (7, 11, 13)])
    g2 = g.copy()
    g2[[7, 11, 13]] = 0.0
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, np.where(np.arange(40) == 13, 0, inp.y), inp.tau, g2)
    assert rel_fro(dX[keep], ref.dX[keep]) <= TOL_GRAD_REL
    for k in range(2):
        assert rel_fro(_np(bw["dW"][k]), ref.dW[k]) <= TOL_GRAD_REL
        assert rel_fro(_np(bw["db"][k]), ref.db[k]) <= TOL_GRAD_REL


def test_binding_rejects_mismatched_extents_before_any_launch(lp):
    # the library sees only pointers: every extent it would read or write is checked first
    import torch
    part = synth.ranges_partition(500, 512, [0, 256, 512])
    T, H = 16, 64
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=9, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    f = lp.lp_forward(X, W, b, P, y, inp.tau)
    g = torch.ones(T, device="cuda")
    bad_cases = [
        lambda: lp.lp_forward(X, [W[0][:, :32].contiguous(), W[1]], b, P, y, inp.tau),   # W of another H
        lambda: lp.lp_forward(X, [W[0][:200].contiguous(), W[1]], b, P, y, inp.tau),     # W short of V_k rows
        lambda: lp.lp_forward(X, W, [b[0][:100].contiguous(), b[1]], P, y, inp.tau),     # bias short
        lambda: lp.lp_forward(X, W, b, P, y[:8].contiguous(), inp.tau),                  # y short
        lambda: lp.lp_top_p_replay(X, W, b, P, torch.full((T, 64), -1, dtype=torch.int32, device="cuda"),
                                   y[:8].contiguous(), inp.tau),
        lambda: lp.lp_backward(X, W, b, P, y, inp.tau, f["lse"][:8].contiguous(), g),     # lse short
        lambda: lp.lp_forward_from_logits([torch.zeros((T, 200), dtype=torch.bfloat16, device="cuda"),
                                           torch.zeros((T, 256), dtype=torch.bfloat16, device="cuda")], P, y,
                                          inp.tau),                                        # logits narrower
        lambda: lp.lp_top_p_replay_dense_mask(X, W, b, P, [torch.zeros((T, 256), dtype=torch.uint8, device="cuda"),
                                                           torch.zeros((T, 100), dtype=torch.uint8,
                                                                       device="cuda")], y, inp.tau),
        lambda: lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True,
                              out={"logp": torch.empty(T, device="cuda"), "lse": torch.empty(T, device="cuda"),
                                   "shard_stats": torch.empty((1, 3, T), device="cuda")}),
    ]
    for i, case in enumerate(bad_cases):
        with pytest.raises(ValueError):
            case()
    assert lp.lp_get_device_error() == 0
