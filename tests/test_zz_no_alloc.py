"""lp_forward_noalloc: the fused forward for callers that cannot allocate device memory
(an engine plugin whose host owns every device byte, a fixed memory budget, no CUDA
allocator binding). It takes its scratch from a fixed array inside the library and runs
the same kernels on the same workspace layout as lp_forward, so it must give lp_forward's
results bit for bit, call after call, even though the array keeps whatever the previous
call left in it.

This file is collected last on purpose; it runs the same alone in a fresh process.
"""
import numpy as np
import pytest

import synth
from lp_util import TOL_ENT, TOL_LOGP, TOL_LSE, dev_inputs, max_abs, part_of

pytestmark = pytest.mark.gpu

KEYS = ("logp", "lse", "entropy", "shard_stats")


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


def _same_bits(lp, got, ref):
    import torch
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), k


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
        _same_bits(lp, got, ref)                           # same kernels, same layout: same bits
        assert max_abs(_np(got["logp"]), _np(ref["logp"])) <= TOL_LOGP
        assert max_abs(_np(got["lse"]), _np(ref["lse"])) <= TOL_LSE
        assert max_abs(_np(got["entropy"]), _np(ref["entropy"])) <= TOL_ENT


def test_noalloc_limit_is_exact_at_the_qwen3_vocabulary(lp):
    """At V = 151936 (594 vocabulary blocks) 4704 rows fit the 32 MiB scratch and 4705 do not;
    the largest accepted batch still gives lp_forward's bits."""
    import torch
    part = synth.even_partition(151936, 1)
    P = part_of(part)
    H = 64
    fits, over = 4704, 4705
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, fits, H, P) <= lp.LP_NOALLOC_SCRATCH_BYTES
    assert lp.lp_workspace_size(lp.LP_OP_FORWARD, over, H, P) > lp.LP_NOALLOC_SCRATCH_BYTES
    inp = synth.forward_inputs(over, H, part, tau=0.7, seed=3, w_std=0.05)
    X, W, _, y = dev_inputs(inp)
    with pytest.raises(lp.LPError) as e:
        lp.lp_forward_noalloc(X, W, None, P, y, inp.tau)
    assert e.value.status == 4                           # LP_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert lp.lp_get_device_error() == 0
    Xf, yf = X[:fits].contiguous(), y[:fits].contiguous()
    ref = lp.lp_forward(Xf, W, None, P, yf, inp.tau, shard_stats=True)
    got = lp.lp_forward_noalloc(Xf, W, None, P, yf, inp.tau, shard_stats=True)
    assert lp.lp_get_device_error() == 0
    _same_bits(lp, got, ref)
    assert torch.isfinite(got["lse"]).all()
