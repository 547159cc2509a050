"""lp_forward_host: rows copied from pinned host memory in chunks that overlap the
forward give the same bits as one lp_forward call on device-resident inputs."""
import pytest

import synth
from lp_util import dev_inputs, part_of

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


@pytest.mark.parametrize("T,chunk", [(3000, 1024), (700, 128), (64, 1024)])
def test_host_forward_is_bitwise_the_device_forward(lp, T, chunk):
    import numpy as np
    import torch
    part = synth.ranges_partition(5000, 5120, [0, 2560, 5120])
    inp = synth.forward_inputs(T, 256, part, tau=0.7, seed=T, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    ref = lp.lp_forward(X, W, b, P, y, inp.tau)
    hX = torch.from_numpy(inp.X.view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.from_numpy(inp.y).pin_memory()
    staging = {}
    for _ in range(2):                      # reuse of the staging buffers across calls
        out = lp.lp_forward_host(hX, W, b, P, hy, inp.tau, chunk_rows=chunk, staging=staging)
        for k in ("logp", "lse", "entropy"):
            assert torch.equal(out[k], ref[k].cpu()), k
    assert lp.lp_get_device_error() == 0
