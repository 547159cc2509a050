"""The vocab_parallel module end to end on a GPU, in a process group of one rank (every GPU
call of this suite has one GPU): the all-gathers, the merge and the ordered sum run through
the module exactly as they would on several ranks. With the rank holding every shard, its
forward is bitwise lp_forward and its autograd gradients are bitwise those of the one-GPU
autograd wrapper."""
import os
import socket

import numpy as np
import pytest

import synth
from lp_util import dev_f32, dev_inputs, part_of

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


@pytest.fixture(scope="module")
def group():
    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("no NCCL in this PyTorch")
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield None
    dist.destroy_process_group()


def test_single_rank_group_forward_and_autograd(lp, group):
    import torch
    from lm_head_linear_tcgen05_gb300 import autograd as ag
    from lm_head_linear_tcgen05_gb300 import vocab_parallel as vp
    part = synth.ranges_partition(6000, 6144, [0, 2048, 4096, 6144])
    P = part_of(part)
    inp = synth.forward_inputs(300, 128, part, tau=0.7, seed=55, w_std=0.05, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    whole = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
    out = vp.forward(X, W, b, P, [0, 1, 2], y, inp.tau, group=group)
    for k in ("logp", "lse", "entropy"):
        assert torch.equal(out[k], whole[k]), k
    # autograd through the module against the one-GPU wrapper
    g = dev_f32(synth.upstream_grad(300, seed=55))
    h = dev_f32(synth.upstream_grad(300, seed=56))

    def run(fn):
        Xr = X.clone().requires_grad_(True)
        Wr = [w.clone().requires_grad_(True) for w in W]
        br = [t.clone().requires_grad_(True) for t in b]
        logp, ent = fn(Xr, Wr, br)
        ((logp * g).sum() + (ent * h).sum()).backward()
        return logp.detach(), ent.detach(), Xr.grad, [w.grad for w in Wr], [t.grad for t in br]

    a = run(lambda Xr, Wr, br: vp.linear_logp(Xr, Wr, br, P, [0, 1, 2], y, inp.tau, group=group))
    r = run(lambda Xr, Wr, br: ag.linear_logp(Xr, Wr, br, P, y, inp.tau))
    assert torch.equal(a[0], r[0]) and torch.equal(a[1], r[1])
    assert torch.equal(a[2], r[2])                        # dX: the one rank's share, rounded once
    for k in range(3):
        assert torch.equal(a[3][k], r[3][k]) and torch.equal(a[4][k], r[4][k])
    # the logits-reuse and replay routes through the module
    L, yl, tau = synth.logits_inputs(300, part, 0.7, seed=57)
    from lp_util import dev_bf16, dev_i32
    Ld = [dev_bf16(t) for t in L]
    yld = dev_i32(yl)
    ol = vp.forward_from_logits(Ld, P, [0, 1, 2], yld, tau, group=group)
    wl = lp.lp_forward_from_logits(Ld, P, yld, tau)
    for k in ("logp", "lse", "entropy"):
        assert torch.equal(ol[k], wl[k]), k
    ids, yr = synth.replay_ids(300, part, seed=58)
    orp = vp.top_p_replay(X, W, b, P, [0, 1, 2], dev_i32(ids), dev_i32(yr), inp.tau, group=group)
    wr = lp.lp_top_p_replay(X, W, b, P, dev_i32(ids), dev_i32(yr), inp.tau)
    assert torch.equal(orp["logp"], wr["logp"]) and torch.equal(orp["lse"], wr["lse"])
    assert lp.lp_get_device_error() == 0
