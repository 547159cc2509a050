"""The entry points issue only stream work once a device is set up, so they can be
captured into a CUDA graph: replaying the graph gives the same bits as the eager call,
and follows new input values written into the captured buffers. Covers inference
(forward, replay, logits reuse) and training (backward options, the logits gradient, and
a whole autograd step)."""
import numpy as np
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


def _capture(fn):
    """Warm up fn on a side stream, then capture one call into a graph."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def test_forward_and_backward_replay_in_a_graph(lp):
    import torch
    part = synth.ranges_partition(5000, 5120, [0, 2560, 5120])
    inp = synth.forward_inputs(300, 256, part, tau=0.7, seed=21, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    g_up = dev_f32(synth.upstream_grad(300, seed=21))
    P = part_of(part)
    ws_f = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, 300, 256, P), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(lp.lp_workspace_size(lp.LP_OP_BACKWARD, 300, 256, P), dtype=torch.uint8, device="cuda")

    def step():
        f = lp.lp_forward(X, W, b, P, y, inp.tau, workspace=ws_f)
        bw = lp.lp_backward(X, W, b, P, y, inp.tau, f["lse"], g_up, workspace=ws_b)
        return f, bw

    graph, (gf, gb) = _capture(step)
    graph.replay()
    torch.cuda.synchronize()
    ef, eb = step()
    torch.cuda.synchronize()
    for k in ("logp", "lse", "entropy"):
        assert torch.equal(gf[k], ef[k]), k
    assert torch.equal(gb["dX"], eb["dX"])
    for k in range(2):
        assert torch.equal(gb["dW"][k], eb["dW"][k]) and torch.equal(gb["db"][k], eb["db"][k])
    # new values in the captured input buffers flow through the replay
    inp2 = synth.forward_inputs(300, 256, part, tau=0.7, seed=22, bias_std=0.1)
    X2, _, _, y2 = dev_inputs(inp2)
    X.copy_(X2)
    y.copy_(y2)
    graph.replay()
    torch.cuda.synchronize()
    ef2, _ = step()
    torch.cuda.synchronize()
    assert torch.equal(gf["logp"], ef2["logp"]) and not torch.equal(ef2["logp"], ef["logp"])
    assert lp.lp_get_device_error() == 0


def test_logits_reuse_and_replay_in_a_graph(lp):
    import torch
    part = synth.even_partition(8192, 4)
    L, yl, tau = synth.logits_inputs(64, part, 0.7, seed=3)
    from lp_util import dev_bf16
    Ld = [dev_bf16(a) for a in L]
    yd = dev_i32(yl)
    ids, yr = synth.replay_ids(64, part, seed=4)
    inp = synth.forward_inputs(64, 128, part, tau=0.7, seed=5)
    X, W, _, _ = dev_inputs(inp)
    ids_d, yr_d = dev_i32(ids), dev_i32(yr)
    P = part_of(part)

    def step():
        a = lp.lp_forward_from_logits(Ld, P, yd, tau)
        r = lp.lp_top_p_replay(X, W, None, P, ids_d, yr_d, tau)
        q = lp.lp_top_p_replay_from_logits(Ld, P, ids_d, yr_d, tau)
        return a, r, q

    graph, (ga, gr, gq) = _capture(step)
    graph.replay()
    torch.cuda.synchronize()
    ea, er, eq = step()
    torch.cuda.synchronize()
    for k in ("logp", "lse", "entropy"):
        assert torch.equal(ga[k], ea[k]), k
    for k in ("logp", "lse"):
        assert torch.equal(gr[k], er[k]) and torch.equal(gq[k], eq[k]), k
    assert lp.lp_get_device_error() == 0


def test_training_step_with_options_in_a_graph(lp):
    # forward, backward with bf16 dX accumulating into caller dW / db, and the logits route
    # with its gradient, all in one graph; two replays equal the same eager sequence bit for bit
    import torch
    part = synth.ranges_partition(3000, 3072, [0, 1536, 3072])
    T, H = 200, 128
    inp = synth.forward_inputs(T, H, part, tau=0.9, seed=31, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    g_up = dev_f32(synth.upstream_grad(T, seed=31))
    h_up = dev_f32(synth.upstream_grad(T, seed=32))
    P = part_of(part)
    L, yl, tau = synth.logits_inputs(T, part, 0.9, seed=33)
    from lp_util import dev_bf16
    Ld = [dev_bf16(a) for a in L]
    yld = dev_i32(yl)
    ws_f = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, P), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(lp.lp_workspace_size(lp.LP_OP_BACKWARD, T, H, P), dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    dW0 = [torch.randn((1536, H), generator=gen, device="cuda") for _ in range(2)]
    db0 = [torch.randn(1536, generator=gen, device="cuda") for _ in range(2)]
    dW = [t.clone() for t in dW0]
    db = [t.clone() for t in db0]
    dL = [torch.empty_like(x) for x in Ld]

    def step():
        f = lp.lp_forward(X, W, b, P, y, inp.tau, workspace=ws_f)
        bw = lp.lp_backward_ex(X, W, b, P, y, inp.tau, f["lse"], g_up, workspace=ws_b, entropy=f["entropy"],
                               grad_entropy=h_up, dx_dtype=torch.bfloat16, accumulate=True, dW=dW, db=db)
        fl = lp.lp_forward_from_logits(Ld, P, yld, tau)
        lp.lp_backward_from_logits(Ld, P, yld, tau, fl["lse"], g_up, entropy=fl["entropy"], grad_entropy=h_up,
                                   out=dL)
        return f, bw

    graph, (gf, gb) = _capture(step)          # the eager warm-up accumulated once ...
    for t, t0 in zip(dW + db, dW0 + db0):     # ... so start the replays from the initial values
        t.copy_(t0)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    got_dW = [t.clone() for t in dW]
    got_db = [t.clone() for t in db]
    got_dX = gb["dX"].clone()
    got_dL = [t.clone() for t in dL]
    for t, t0 in zip(dW + db, dW0 + db0):
        t.copy_(t0)
    step()
    e = step()[1]
    torch.cuda.synchronize()
    assert torch.equal(got_dX, e["dX"]) and got_dX.dtype == torch.bfloat16
    for a, c in zip(got_dW + got_db, dW + db):
        assert torch.equal(a, c)
    for a, c in zip(got_dL, dL):
        assert torch.equal(a, c)
    assert lp.lp_get_device_error() == 0


def test_autograd_step_in_a_graph(lp):
    # a whole autograd step (forward, loss, backward into .grad) captured and replayed
    import torch
    from lm_head_linear_tcgen05_gb300.autograd import linear_logp
    part = synth.ranges_partition(2000, 2048, [0, 1024, 2048])
    T, H = 130, 64
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=41, w_std=0.2, bias_std=0.05)
    X0, W0, b0, y = dev_inputs(inp)
    X = X0.clone().requires_grad_(True)
    W = [w.clone().requires_grad_(True) for w in W0]
    P = part_of(part)
    a = dev_f32(synth.upstream_grad(T, seed=42))
    c = dev_f32(synth.upstream_grad(T, seed=43))

    def step():
        logp, ent = linear_logp(X, W, None, P, y, inp.tau)
        ((logp * a).sum() + (ent * c).sum()).backward()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            X.grad = None
            for w in W:
                w.grad = None
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    X.grad = None
    for w in W:
        w.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    gX = X.grad.clone()
    gW = [w.grad.clone() for w in W]
    X.grad = None
    for w in W:
        w.grad = None
    step()
    torch.cuda.synchronize()
    assert torch.equal(gX, X.grad)
    for u, w in zip(gW, W):
        assert torch.equal(u, w.grad)
