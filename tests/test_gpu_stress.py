"""Repetition stress: hundreds of back-to-back calls of every kernel on one stream, each
result compared bit for bit with the first. A race (a read that overtakes a write, a
barrier phase reused too early, a slot claimed twice) would show up as a flipped bit in
some call long before it shows up against the oracle's tolerances."""
import pytest

import synth
from lp_util import dev_f32, dev_i32, dev_inputs, part_of

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


def _same(a, b):
    import torch
    if isinstance(a, dict):
        return all(_same(a[k], b[k]) for k in a if a[k] is not None)
    if isinstance(a, (list, tuple)):
        return all(_same(x, y) for x, y in zip(a, b) if x is not None)
    return torch.equal(a, b)


def test_every_kernel_repeats_bit_for_bit(lp):
    import torch
    part = synth.ranges_partition(30000, 30208, [0, 10112, 20160, 30208])   # padding in the last shard
    T, H = 1000, 1024
    inp = synth.forward_inputs(T, H, part, tau=0.8, seed=123, w_std=0.05, bias_std=0.05)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    g = dev_f32(synth.upstream_grad(T, seed=124))
    h = dev_f32(synth.upstream_grad(T, seed=125))
    ids, yr = synth.replay_ids(T, part, seed=126)
    ids_d, yr_d = dev_i32(ids), dev_i32(yr)
    L = [torch.randn((T, e - s), generator=torch.Generator(device="cuda").manual_seed(k), device="cuda")
         .mul(3).to(torch.bfloat16) for k, (s, e) in enumerate(part.ranges)]
    ws_f = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, P), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(lp.lp_workspace_size(lp.LP_OP_BACKWARD, T, H, P), dtype=torch.uint8, device="cuda")

    fwd = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True, workspace=ws_f)
    calls = {
        "forward": lambda: lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True, workspace=ws_f),
        "backward": lambda: lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], g, workspace=ws_b, entropy=fwd["entropy"],
                                           grad_entropy=h),
        "logits": lambda: lp.lp_forward_from_logits(L, P, y, inp.tau, shard_stats=True),
        "logits_grad": lambda: lp.lp_backward_from_logits(L, P, y, inp.tau, fwd["lse"], g),
        "replay": lambda: lp.lp_top_p_replay(X, W, b, P, ids_d, yr_d, inp.tau, shard_stats=True),
        "replay_logits": lambda: lp.lp_top_p_replay_from_logits(L, P, ids_d, yr_d, inp.tau),
    }
    reps = {"forward": 300, "backward": 60, "logits": 300, "logits_grad": 200, "replay": 300, "replay_logits": 300}
    for name, fn in calls.items():
        first = fn()
        outs = [fn() for _ in range(reps[name])]   # enqueued back to back, compared afterwards
        torch.cuda.synchronize()
        for i, o in enumerate(outs):
            assert _same(first, o), (name, i)
        del outs
    assert lp.lp_get_device_error() == 0
