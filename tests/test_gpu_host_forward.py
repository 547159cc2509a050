"""lp_forward_host (the C entry point on host-resident rows): its results are bitwise those
of lp_forward on device-resident inputs, with page-locked or pageable host buffers, with
every optional output, with reused workspace and output buffers, for an empty batch, and
for batches of 4096 rows and more, which run as two halves whose second half is copied in
on another stream while the first computes (ragged halves included)."""
import numpy as np
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


@pytest.mark.parametrize("T,pinned", [(3000, True), (700, False), (64, True), (4096, True), (5001, True),
                                      (4099, False)])
def test_host_forward_is_bitwise_the_device_forward(lp, T, pinned):
    import torch
    part = synth.ranges_partition(5000, 5120, [0, 2560, 2560, 5120])     # an empty shard, padding
    inp = synth.forward_inputs(T, 256, part, tau=0.7, seed=T, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    ref = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
    hX = torch.from_numpy(inp.X.view(np.int16)).view(torch.bfloat16)
    hy = torch.from_numpy(inp.y)
    if pinned:
        hX, hy = hX.pin_memory(), hy.pin_memory()
    ws = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD_HOST, T, 256, P), dtype=torch.uint8, device="cuda")
    out = None
    for _ in range(2):                      # reuse of the workspace and the host outputs
        got = lp.lp_forward_host(hX, W, b, P, hy, inp.tau, shard_stats=True, workspace=ws, out=out)
        out = got
        for k in ("logp", "lse", "entropy", "shard_stats"):
            assert not got[k].is_cuda and torch.equal(got[k], ref[k].cpu()), k
    # optional outputs off
    got = lp.lp_forward_host(hX, W, b, P, hy, inp.tau, entropy=False)
    assert got["entropy"] is None and got["shard_stats"] is None
    assert torch.equal(got["logp"], ref["logp"].cpu()) and torch.equal(got["lse"], ref["lse"].cpu())
    assert lp.lp_get_device_error() == 0


def test_host_forward_empty_batch_and_errors(lp):
    import torch
    part = synth.even_partition(1000, 1)
    inp = synth.forward_inputs(8, 64, part, tau=0.7, seed=2)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    hX = torch.from_numpy(inp.X.view(np.int16)).view(torch.bfloat16)
    hy = torch.from_numpy(inp.y)
    e = lp.lp_forward_host(hX[:0], W, b, P, hy[:0], inp.tau)
    assert e["logp"].shape == (0,)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lp.LPError, match="WORKSPACE_TOO_SMALL"):
        lp.lp_forward_host(hX, W, b, P, hy, inp.tau, workspace=small)
    with pytest.raises(ValueError):
        lp.lp_forward_host(X, W, b, P, hy, inp.tau)                      # device tensors are not host rows
    with pytest.raises(ValueError):
        lp.lp_forward_host(hX, W, b, P, hy[:4].contiguous(), inp.tau)     # y of another length
    assert lp.lp_get_device_error() == 0


def test_host_forward_from_concurrent_threads(lp):
    """Two host threads, each on its own stream with its own workspace and host buffers,
    call lp_forward_host on two-part batches at the same time: the calls share the
    device's copy stream and events, and every result is still bitwise lp_forward's."""
    import threading

    import torch
    part = synth.ranges_partition(2000, 2048, [0, 1024, 2048])
    P = part_of(part)
    cases = []
    for i, T in enumerate((4096, 4357)):
        inp = synth.forward_inputs(T, 256, part, tau=0.7, seed=40 + i, bias_std=0.1)
        X, W, b, y = dev_inputs(inp)
        ref = lp.lp_forward(X, W, b, P, y, inp.tau, shard_stats=True)
        hX = torch.from_numpy(inp.X.view(np.int16)).view(torch.bfloat16).pin_memory()
        hy = torch.from_numpy(inp.y).pin_memory()
        ws = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD_HOST, T, 256, P), dtype=torch.uint8,
                         device="cuda")
        cases.append((hX, W, b, hy, inp.tau, ws, {k: ref[k].cpu() for k in ref if ref[k] is not None}))
    torch.cuda.synchronize()
    failures = []

    def worker(case):
        hX, W, b, hy, tau, ws, ref = case
        torch.cuda.set_device(0)
        with torch.cuda.stream(torch.cuda.Stream()):
            out = None
            for it in range(25):
                got = lp.lp_forward_host(hX, W, b, P, hy, tau, shard_stats=True, workspace=ws, out=out)
                out = got
                for k in ("logp", "lse", "entropy", "shard_stats"):
                    if not torch.equal(got[k], ref[k]):
                        failures.append((hX.shape[0], it, k))

    threads = [threading.Thread(target=worker, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not failures, failures[:5]
    assert lp.lp_get_device_error() == 0
