"""lp_forward_noalloc: the fused forward for callers that cannot allocate device memory
(an engine plugin whose host owns every device byte, a fixed memory budget, no CUDA
allocator binding). It takes its scratch from a fixed array inside the library, so it
must give the same results as lp_forward with a caller workspace, call after call,
even though the array keeps whatever the previous call left in it.

This file is collected last on purpose; it runs the same alone in a fresh process.
"""
import numpy as np
import pytest

import synth
from lp_util import TOL_ENT, TOL_LOGP, TOL_LSE, dev_inputs, max_abs, part_of

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


def test_noalloc_matches_lp_forward_on_two_calls_in_a_row(lp):
    cases = [
        # (T, H, bounds, vocab_real, bias_std, seed)
        (700, 256, [0, 3000, 3000, 7000, 8192], 8000, 0.2, 1),
        (129, 192, [0, 5000], 5000, None, 2),
    ]
    for T, H, bounds, real, bias, seed in cases:          # two calls, different shapes and data
        part = synth.ranges_partition(real, bounds[-1], bounds)
        inp = synth.forward_inputs(T, H, part, tau=0.7, seed=seed, w_std=0.05, bias_std=bias)
        X, W, b, y = dev_inputs(inp)
        P = part_of(part)
        ref = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
        got = lp.lp_forward_noalloc(X, W, b, P, y, inp.tau, shard_stats=True)
        assert lp.lp_get_device_error() == 0
        assert max_abs(_np(got["logp"]), _np(ref["logp"])) <= TOL_LOGP
        assert max_abs(_np(got["lse"]), _np(ref["lse"])) <= TOL_LSE
        assert max_abs(_np(got["entropy"]), _np(ref["entropy"])) <= TOL_ENT
        ss_g, ss_r = _np(got["shard_stats"]), _np(ref["shard_stats"])
        assert max_abs(ss_g[:, 0], ss_r[:, 0]) <= TOL_LSE
        assert max_abs(ss_g[:, 1], ss_r[:, 1]) <= TOL_LOGP
        assert max_abs(ss_g[:, 2], ss_r[:, 2]) <= TOL_ENT


def test_noalloc_rejects_problems_beyond_its_scratch(lp):
    import torch
    part = synth.even_partition(151936, 1)
    P = part_of(part)
    T, H = 6000, 64
    need = lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, P)
    assert need > lp.LP_NOALLOC_SCRATCH_BYTES
    X = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    W = [torch.zeros((151936, H), dtype=torch.bfloat16, device="cuda")]
    y = torch.zeros(T, dtype=torch.int32, device="cuda")
    with pytest.raises(lp.LPError) as e:
        lp.lp_forward_noalloc(X, W, None, P, y, 0.7)
    assert e.value.status == 4                           # LP_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert lp.lp_get_device_error() == 0
