"""Failure detection without a GPU fault: a bounded pipeline wait that nothing will
satisfy gives up, reports LP_ERR_DEVICE_TIMEOUT through the device error word and
leaves the context usable for the next call."""
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
