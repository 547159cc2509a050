"""Host logic of the multi-GPU benchmark run (replicas, weak scaling), on CPU with two
gloo ranks: the only collective is the max of the per-rank step times, and the
whole-job rate counts every rank's rows over the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max_ms(1.0 + 0.5 * rank, dist, "cpu")
        out[rank] = (ms, bench.whole_job_rate(4096, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, rate = res[r]
        assert ms == 1.5
        assert rate == pytest.approx(2 * 4096 / 1.5e-3)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.reduce_max_ms(2.5, None, "cpu") == 2.5
    assert bench.whole_job_rate(4096, 1, 2.0) == pytest.approx(4096 / 2e-3)
