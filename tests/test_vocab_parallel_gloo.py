"""Host side of the vocabulary-parallel exchange on CPU, with two gloo ranks: each rank
contributes the statistics of its own shards (rank 0 three shards, rank 1 one) and its
share of dX; the all-gathers give every rank the same bytes in rank order, and folding
them gives the unsharded result. The statistics and shares come from the oracle here
(the library's own merge and ordered sum are exercised on the GPU); what is tested is the
exchange itself - completeness, order, identical results on every rank."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

BOUNDS = [0, 100, 250, 380, 512]
REAL = 500
RANK_SHARDS = {0: [0, 1, 2], 1: [3]}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem():
    part = synth.ranges_partition(REAL, BOUNDS[-1], BOUNDS)
    inp = synth.forward_inputs(24, 32, part, tau=0.7, seed=21, w_std=0.2, bias_std=0.1)
    return part, inp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    from lm_head_linear_tcgen05_gb300 import vocab_parallel as vp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        part, inp = _problem()
        y = inp.y.astype(np.int64)
        z = oracle.logits_from_bits(inp.X, inp.W, inp.bias, part, inp.tau)
        st = oracle.shard_stats(z, y, part.ranges, part.vocab_real)
        mine = RANK_SHARDS[rank]
        local = torch.tensor(np.stack([np.stack([st[k].lse, st[k].t, st[k].h]) for k in mine]), dtype=torch.float32)
        gathered = vp.gather_shard_stats(local)
        # this rank's share of dX: the oracle backward restricted to its shards
        g = synth.upstream_grad(24, seed=21)
        full = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, g)
        Wd = [oracle.bf16_to_f64(w) for w in inp.W]
        G = _g_matrix(z, y, inp.tau, g, part)
        share = sum(G[k] @ Wd[k] for k in mine).astype(np.float32)
        shares = vp.gather_in_rank_order(torch.from_numpy(share)[None])
        out[rank] = (gathered.numpy().copy(), np.concatenate([s.numpy() for s in shares]), full.dX)
    finally:
        dist.destroy_process_group()


def _g_matrix(z, y, tau, g, part):
    """Per shard, the rows x local ids block of G = g (onehot - p) / tau (0 on padding)."""
    M = z.max(axis=1, keepdims=True)
    p = np.exp(z - M)
    p /= p.sum(axis=1, keepdims=True)
    G = -p
    G[np.arange(z.shape[0]), y] += 1.0
    G *= (g / tau)[:, None]
    out = []
    for s, e in part.ranges:
        Gk = np.zeros((z.shape[0], e - s))
        hi = min(e, part.vocab_real)
        Gk[:, : hi - s] = G[:, s:hi]
        out.append(Gk)
    return out


def test_two_gloo_ranks_exchange_statistics_and_dx_shares_in_rank_order():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    part, inp = _problem()
    y = inp.y.astype(np.int64)
    z = oracle.logits_from_bits(inp.X, inp.W, inp.bias, part, inp.tau)
    st = oracle.shard_stats(z, y, part.ranges, part.vocab_real)
    expect = np.stack([np.stack([s.lse, s.t, s.h]) for s in st]).astype(np.float32)
    g0, sh0, dx = res[0]
    g1, sh1, _ = res[1]
    # every rank holds the same bytes: all four shards, in ascending (rank) order
    assert g0.shape == (4, 3, 24)
    assert g0.tobytes() == g1.tobytes() == expect.tobytes()
    assert sh0.tobytes() == sh1.tobytes() and sh0.shape == (2, 24, 32)
    # folding the gathered statistics gives the unsharded softmax
    dense = oracle.forward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau)
    logp, lse, ent = oracle.merge_shard_stats(g0[:, 0], g0[:, 1], g0[:, 2], y, part.ranges, part.vocab_real)
    np.testing.assert_allclose(lse, dense.lse, atol=1e-5)
    np.testing.assert_allclose(ent, dense.entropy, atol=1e-5)
    np.testing.assert_allclose(logp, dense.logp, atol=1e-5)
    # the rank-ordered sum of the dX shares is the whole dX
    acc = sh0[0].copy()
    acc += sh0[1]
    np.testing.assert_allclose(acc, dx, rtol=1e-5, atol=1e-6)


def test_rank_partition_is_a_local_run_of_shards():
    from lm_head_linear_tcgen05_gb300 import VocabPartition
    from lm_head_linear_tcgen05_gb300 import vocab_parallel as vp
    full = VocabPartition(REAL, BOUNDS[-1], tuple(zip(BOUNDS[:-1], BOUNDS[1:])))
    p = vp.rank_partition(full, [1, 2])
    assert p.local and p.ranges == ((100, 250), (250, 380)) and p.vocab_real == REAL
    with pytest.raises(ValueError):
        vp.rank_partition(full, [0, 2])
    with pytest.raises(ValueError):
        vp.rank_partition(full, [])
    with pytest.raises(ValueError):
        vp.rank_partition(full, [4])
