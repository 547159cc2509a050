"""GPU parity of the fused forward against the fp64 oracle, bitwise determinism, batch
invariance, closed forms and the device-side error path (all through the C ABI)."""
import math

import numpy as np
import pytest

import oracle
import synth
from lp_util import (TOL_ENT, TOL_LOGP, TOL_LSE, dev_bf16, dev_i32, dev_inputs, max_abs, part_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lp():
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    import lm_head_linear_tcgen05_gb300 as mod
    import torch
    assert mod.lp_device_supported(), "current device cannot run liblp.so"
    torch.cuda.set_device(0)
    return mod


def _np(t):
    return t.detach().cpu().numpy()


def _run(lp, inp, **kw):
    X, W, b, y = dev_inputs(inp)
    out = lp.lp_forward(X, W, b, part_of(inp.part), y, inp.tau, **kw)
    assert lp.lp_get_device_error() == 0
    return out


def _compare(out, ref, shard_stats=False):
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE
    assert max_abs(_np(out["entropy"]), ref.entropy) <= TOL_ENT
    if shard_stats:
        ss = _np(out["shard_stats"])
        for k, s in enumerate(ref.shards):
            assert max_abs(ss[k, 0], s.lse) <= TOL_LSE
            assert max_abs(ss[k, 1], s.t) <= TOL_LOGP
            assert max_abs(ss[k, 2], s.h) <= TOL_ENT


def test_tiny_config_parity(lp):
    # T=64, H=256, V=1000, one shard, no bias, tau=1.0
    part = synth.even_partition(1000, 1)
    inp = synth.forward_inputs(64, 256, part, tau=1.0, seed=0)
    out = _run(lp, inp, shard_stats=True)
    ref = oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    _compare(out, ref, shard_stats=True)


@pytest.mark.parametrize("T,H,bounds,real,bias", [
    (300, 192, [0, 300, 300, 700, 1024], 1000, 0.5),    # ragged rows, K tail (192 % 64 = 0, 192 < 256), empty shard, padding
    (129, 200, [0, 1000], 999, None),                  # H not a multiple of 64, one padded id
    (1, 64, [0, 513, 777, 2100], 2048, 0.3),           # single row, odd shard widths, padded tail spans shards
    (257, 520, [0, 256, 512], 512, None),              # exact tiles
])
def test_sharded_padded_parity(lp, T, H, bounds, real, bias):
    part = synth.ranges_partition(real, bounds[-1], bounds)
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=T + H, w_std=0.05, bias_std=bias)
    out = _run(lp, inp, shard_stats=True)
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    _compare(out, ref, shard_stats=True)


def test_w_zero_closed_form_with_padding(lp):
    # z == 0 on the real ids: logp = -log V_real exactly up to exp/log rounding; the
    # 128 padded ids would shift it by 8.4e-4, so the bound here is 1e-5
    part = synth.ranges_partition(151936 // 16, 152064 // 16, [0, 2376, 4752, 7128, 9504])
    T, H = 130, 64
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=1)
    inp.W = [np.zeros_like(w) for w in inp.W]
    out = _run(lp, inp)
    v = part.vocab_real
    assert max_abs(_np(out["logp"]), np.full(T, -math.log(v))) <= 1e-5
    assert max_abs(_np(out["lse"]), np.full(T, math.log(v))) <= 1e-5
    assert max_abs(_np(out["entropy"]), np.full(T, math.log(v))) <= 1e-5


def test_one_dominant_logit(lp):
    part = synth.even_partition(4096, 2)
    T, H, tau = 8, 64, 1.0
    inp = synth.forward_inputs(T, H, part, tau=tau, seed=2)
    inp.W = [np.zeros_like(w) for w in inp.W]
    inp.y[:] = 3001                       # the bias is shared by all rows: one hot id
    hot = np.zeros(4096, np.float32)
    hot[3001] = 100.0
    inp.bias = [synth.bf16_bits(hot[:2048]), synth.bf16_bits(hot[2048:])]
    out = _run(lp, inp)
    assert np.all(np.abs(_np(out["logp"])) <= 1e-5)
    assert np.all(np.abs(_np(out["entropy"])) <= 1e-3)


def test_bitwise_repeatable(lp):
    part = synth.ranges_partition(3000, 3072, [0, 1000, 3072])
    inp = synth.forward_inputs(700, 256, part, tau=0.7, seed=5, bias_std=0.1)
    a = _run(lp, inp, shard_stats=True)
    b = _run(lp, inp, shard_stats=True)
    for k in ("logp", "lse", "entropy", "shard_stats"):
        assert np.array_equal(_np(a[k]).view(np.uint32), _np(b[k]).view(np.uint32)), k


def test_batch_invariance_split_and_permute(lp):
    import torch
    part = synth.ranges_partition(5000, 5120, [0, 2560, 5120])
    inp = synth.forward_inputs(1000, 320, part, tau=0.7, seed=6, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    full = lp.lp_forward(X, W, b, P, y, inp.tau)
    # in pieces of 512, 300 and 188 rows
    pieces = []
    for s, e in [(0, 512), (512, 812), (812, 1000)]:
        pieces.append(lp.lp_forward(X[s:e].contiguous(), W, b, P, y[s:e].contiguous(), inp.tau))
    for key in ("logp", "lse", "entropy"):
        cat = torch.cat([p[key] for p in pieces])
        assert torch.equal(cat, full[key]), key
    # batches of at most 128 rows (one row block: these run without clusters) give the same bits
    for s, e in [(0, 1), (5, 133), (700, 797), (872, 1000)]:
        q = lp.lp_forward(X[s:e].contiguous(), W, b, P, y[s:e].contiguous(), inp.tau, shard_stats=True)
        for key in ("logp", "lse", "entropy"):
            assert torch.equal(q[key], full[key][s:e]), (s, e, key)
    # rows permuted
    perm = torch.randperm(1000, generator=torch.Generator().manual_seed(0)).cuda()
    pr = lp.lp_forward(X[perm].contiguous(), W, b, P, y[perm].contiguous(), inp.tau)
    for key in ("logp", "lse", "entropy"):
        assert torch.equal(pr[key], full[key][perm]), key
    assert lp.lp_get_device_error() == 0


def test_target_out_of_range_is_a_device_error(lp):
    part = synth.even_partition(1000, 1)
    inp = synth.forward_inputs(16, 64, part, tau=0.7, seed=7)
    X, W, b, y = dev_inputs(inp)
    y[3] = 1000
    y[5] = -1
    out = lp.lp_forward(X, W, b, part_of(part), y, inp.tau)
    assert lp.lp_get_device_error() == 5
    lg = _np(out["logp"])
    assert np.isneginf(lg[3]) and np.isneginf(lg[5])
    assert np.all(np.isfinite(np.delete(lg, [3, 5])))
    assert not np.any(np.isnan(_np(out["lse"])))
    assert lp.lp_get_device_error() == 0          # cleared by the read


def test_empty_batch_is_a_no_op(lp):
    import torch
    part = synth.even_partition(1000, 2)
    P = part_of(part)
    X = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = [torch.zeros((500, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y = torch.empty(0, dtype=torch.int32, device="cuda")
    out = lp.lp_forward(X, W, None, P, y, 0.7)
    assert out["logp"].numel() == 0
    g = torch.empty(0, dtype=torch.float32, device="cuda")
    bw = lp.lp_backward(X, W, None, P, y, 0.7, out["lse"], g)
    assert all(torch.count_nonzero(d) == 0 for d in bw["dW"]) and all(torch.count_nonzero(d) == 0 for d in bw["db"])
    ids = torch.empty((0, 64), dtype=torch.int32, device="cuda")
    assert lp.lp_top_p_replay(X, W, None, P, ids, y, 0.7)["lse"].numel() == 0
    assert lp.lp_get_device_error() == 0


def test_single_real_id(lp):
    # one real id, the rest padding: every row has logp = 0, LSE = z, entropy = 0
    part = synth.ranges_partition(1, 300, [0, 1, 300])
    inp = synth.forward_inputs(5, 64, part, tau=0.7, seed=8, w_std=0.3, bias_std=0.2)
    inp.y[:] = 0
    out = _run(lp, inp, shard_stats=True)
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    assert np.all(np.abs(_np(out["logp"])) <= 1e-6)      # 0 up to the base-2 rescaling rounding
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE
    assert np.all(np.abs(_np(out["entropy"])) <= 1e-6)
    ss = _np(out["shard_stats"])
    assert np.all(np.isneginf(ss[1, 0])) and np.all(ss[1, 1] == 0)     # the all-padding shard is empty


@pytest.mark.parametrize("tau", [0.05, 20.0])
def test_extreme_temperatures(lp, tau):
    part = synth.ranges_partition(3000, 3072, [0, 1500, 3072])
    inp = synth.forward_inputs(130, 128, part, tau=tau, seed=9, w_std=0.05, bias_std=0.1)
    out = _run(lp, inp)
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    # logits scale as 1/tau: the absolute tolerance applies to z-sized quantities
    scale = max(1.0, 1.0 / tau)
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP * scale
    assert max_abs(_np(out["lse"]), ref.lse) <= TOL_LSE * scale
    assert max_abs(_np(out["entropy"]), ref.entropy) <= TOL_ENT * scale


def test_largest_hidden_size(lp):
    # H = 65536, the largest the library accepts (the replay stages x in 128 KB of shared memory)
    part = synth.even_partition(600, 2)
    inp = synth.forward_inputs(3, 65536, part, tau=0.7, seed=10, w_std=0.004)
    out = _run(lp, inp)
    ref = oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    assert max_abs(_np(out["logp"]), ref.logp) <= TOL_LOGP
    assert max_abs(_np(out["entropy"]), ref.entropy) <= TOL_ENT
    ids, yr = synth.replay_ids(3, part, seed=11)
    X, W, _, _ = dev_inputs(inp)
    rep = lp.lp_top_p_replay(X, W, None, part_of(part), dev_i32(ids), dev_i32(yr), inp.tau)
    rref = oracle.top_p_replay(inp.X, inp.W, None, part, ids, yr, inp.tau)
    assert lp.lp_get_device_error() == 0
    assert max_abs(_np(rep["lse"]), rref.lse) <= TOL_LSE
