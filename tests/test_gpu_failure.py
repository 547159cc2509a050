"""Failure detection without a GPU fault: a bounded pipeline wait that nothing will
satisfy, or a wait given a limit too short to be met, gives up, reports
LP_ERR_DEVICE_TIMEOUT through the device error word and leaves the context usable for the
next call."""
import numpy as np
import pytest

import oracle
import synth
from lp_util import TOL_LOGP, dev_inputs, max_abs, part_of

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


def test_wait_gives_up_and_context_stays_usable(lp):
    assert lp.lp_get_device_error() == 0
    lp.lp_selftest_wait_timeout(5_000_000)              # 5 ms limit on a barrier nothing arrives on
    assert lp.lp_get_device_error() == 7                 # LP_ERR_DEVICE_TIMEOUT
    assert lp.lp_get_device_error() == 0                 # read clears it
    part = synth.even_partition(1000, 1)
    inp = synth.forward_inputs(32, 64, part, tau=0.7, seed=3)
    X, W, b, y = dev_inputs(inp)
    out = lp.lp_forward(X, W, b, part_of(part), y, inp.tau)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    assert max_abs(out["logp"].cpu().numpy(), ref.logp) <= TOL_LOGP


def test_selftest_rejects_unbounded_limits(lp):
    with pytest.raises(lp.LPError):
        lp.lp_selftest_wait_timeout(10_000_000_000)      # 10 s is beyond the 2 s cap


def test_pipeline_waits_give_up_at_a_tiny_limit_and_the_context_stays_usable(lp):
    """The real GEMM pipelines with a 1 us wait limit - far shorter than the K loop of a tile
    at H = 16384 (256 K steps), so at least the epilogue's first wait gives up: a CTA-pair
    forward (T = 256), a single-CTA forward (T = 64) and the backward's three GEMMs each report
    LP_ERR_DEVICE_TIMEOUT and return; at the default limit the same calls are correct again."""
    import torch
    from lp_util import TOL_GRAD_REL, dev_f32, rel_fro
    part = synth.ranges_partition(2000, 2048, [0, 1024, 2048])
    P = part_of(part)
    T0, H = 256, 16384
    inp = synth.forward_inputs(T0, H, part, tau=0.7, seed=5, w_std=0.01, bias_std=0.01)
    X, W, b, y = dev_inputs(inp)
    g = dev_f32(synth.upstream_grad(T0, seed=5))
    lse = torch.zeros(T0, dtype=torch.float32, device="cuda")
    assert lp.lp_get_device_error() == 0
    got = []
    lp.lp_set_wait_limit(1000)
    try:
        for T in (T0, 64):
            lp.lp_forward(X[:T].contiguous(), W, b, P, y[:T].contiguous(), inp.tau)
            got.append(lp.lp_get_device_error())
        lp.lp_backward(X, W, b, P, y, inp.tau, lse, g)
        got.append(lp.lp_get_device_error())
    finally:
        lp.lp_set_wait_limit(0)                          # back to the 2 s default
    assert got == [7, 7, 7]                              # LP_ERR_DEVICE_TIMEOUT each time
    out = lp.lp_forward(X, W, b, P, y, inp.tau)
    bw = lp.lp_backward(X, W, b, P, y, inp.tau, out["lse"], g)
    assert lp.lp_get_device_error() == 0
    ref = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    assert max_abs(out["logp"].cpu().numpy(), ref.logp) <= TOL_LOGP
    rb = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, synth.upstream_grad(T0, seed=5))
    assert rel_fro(bw["dX"].cpu().numpy(), rb.dX) <= TOL_GRAD_REL


def test_wait_limit_setter_rejects_out_of_range_limits(lp):
    with pytest.raises(lp.LPError):
        lp.lp_set_wait_limit(999)
    with pytest.raises(lp.LPError):
        lp.lp_set_wait_limit(10_000_000_001)
    lp.lp_set_wait_limit(0)
