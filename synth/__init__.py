"""Seeded synthetic inputs for the linear-logp operator.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds none of the operator's arithmetic: it only draws random numbers, rounds
them to bf16 storage and lays out vocabulary partitions. Everything it returns is
plain numpy on the host (bf16 tensors as their raw uint16 bit patterns), so the
CUDA path and the oracle consume the very same bits.

Workload recipes (all synthetic stand-ins for the Qwen3-8B LM head used by the
pages "feat(rl-kernel): add CUDA linear logp provider integration" (200-step
reference result) and "Perf/cuda compact top p replay" (Performance)):

* forward: X ~ N(0,1), W ~ N(0, 0.02^2), optional bias ~ N(0, bias_std^2),
  targets uniform over the real vocabulary;
* logits reuse: L ~ N(0, 3^2) with a fraction of entries per row set to +8;
* compact top-p replay: per row 1..64 distinct ids (a nucleus of a Zipf(1.1)
  ranking mapped to vocabulary ids by a per-row random permutation), ~10 %
  duplicate slots, -1 padding, 25 % of rows with one shard left empty, target
  drawn from the row's ids;
* backward: upstream gradient g ~ N(0,1) per row.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

REPLAY_SLOTS = 64


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    # round-to-nearest-even on the 16 dropped bits; NaN never occurs in these inputs
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk_rows: int = 8192) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16, drawn in row chunks to bound peak memory."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        blk = rng.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            blk *= np.float32(std)
        out[r0:r1] = bf16_bits(blk)
    return out


@dataclass(frozen=True)
class Partition:
    """Contiguous vocabulary shards in ascending order covering [0, vocab_padded).

    Ids at or above ``vocab_real`` are padding and never part of the softmax.
    """
    vocab_real: int
    vocab_padded: int
    ranges: Tuple[Tuple[int, int], ...]

    @property
    def n_shards(self) -> int:
        return len(self.ranges)

    def widths(self) -> List[int]:
        return [e - s for s, e in self.ranges]


def even_partition(vocab_real: int, n_shards: int, vocab_padded: Optional[int] = None) -> Partition:
    """Split [0, vocab_padded) into ``n_shards`` equal contiguous shards."""
    vp = vocab_real if vocab_padded is None else vocab_padded
    if vp % n_shards:
        raise ValueError("padded vocabulary must divide evenly into shards")
    w = vp // n_shards
    return Partition(vocab_real, vp, tuple((k * w, (k + 1) * w) for k in range(n_shards)))


def ranges_partition(vocab_real: int, vocab_padded: int, bounds: Sequence[int]) -> Partition:
    """Partition from ascending shard boundaries [b0=0, b1, ..., bK=vocab_padded] (empty shards allowed)."""
    b = list(bounds)
    return Partition(vocab_real, vocab_padded, tuple((b[i], b[i + 1]) for i in range(len(b) - 1)))


@dataclass
class ForwardInputs:
    X: np.ndarray                 # uint16 bf16 bits [T, H]
    W: List[np.ndarray]           # per shard uint16 bf16 bits [V_k, H]
    bias: Optional[List[np.ndarray]]  # per shard uint16 bf16 bits [V_k] or None
    y: np.ndarray                 # int32 [T] global target ids
    tau: float
    part: Partition


def forward_inputs(T: int, H: int, part: Partition, tau: float, seed: int = 0,
                   w_std: float = 0.02, x_std: float = 1.0,
                   bias_std: Optional[float] = None) -> ForwardInputs:
    """X ~ N(0,x_std^2), W ~ N(0,w_std^2) per shard, bias ~ N(0,bias_std^2) (None: no bias), y ~ U[0,V_real)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    X = _normal_bf16(rng, (T, H), x_std)
    W = [_normal_bf16(rng, (e - s, H), w_std) for s, e in part.ranges]
    bias = None
    if bias_std is not None:
        bias = [bf16_bits(rng.standard_normal(e - s, dtype=np.float32) * np.float32(bias_std))
                for s, e in part.ranges]
    y = rng.integers(0, part.vocab_real, size=T, dtype=np.int64).astype(np.int32)
    return ForwardInputs(X, W, bias, y, float(np.float32(tau)), part)


def logits_inputs(T: int, part: Partition, tau: float, seed: int = 0, std: float = 3.0,
                  peak_frac: float = 0.01, peak_value: float = 8.0):
    """Unscaled logits per shard: N(0,std^2) bf16, and per row ``peak_frac`` of the real
    vocabulary (positions uniform without replacement) set to ``peak_value``.

    Returns (list of uint16 [T, V_k] arrays, y int32 [T], tau)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    V = part.vocab_padded
    full = _normal_bf16(rng, (T, V), std, chunk_rows=1024)
    n_peak = int(round(peak_frac * part.vocab_real))
    if n_peak:
        pk = bf16_bits(np.array([peak_value], np.float32))[0]
        for t in range(T):
            cols = rng.choice(part.vocab_real, size=n_peak, replace=False)
            full[t, cols] = pk
    y = rng.integers(0, part.vocab_real, size=T, dtype=np.int64).astype(np.int32)
    shards = [np.ascontiguousarray(full[:, s:e]) for s, e in part.ranges]
    return shards, y, float(np.float32(tau))


def replay_ids(T: int, part: Partition, seed: int = 0, max_ids: int = REPLAY_SLOTS,
               dup_frac: float = 0.10, empty_shard_frac: float = 0.25, zipf_s: float = 1.1):
    """Compact top-p replay sets: int32 [T, 64] slots (-1 = unused) and targets y [T].

    Per row a count c ~ U{1..max_ids} of distinct ids: the c highest-probability
    ranks of a Zipf(zipf_s) ranking (the finite nucleus), mapped to vocabulary ids
    by a per-row random permutation of the real vocabulary. For
    ``empty_shard_frac`` of the rows one random shard is excluded from that
    mapping, so the row has no candidate there. round(dup_frac*c) duplicate
    slots are added (total capped at 64), slots are shuffled and padded with -1.
    The target is drawn uniformly from the row's distinct ids.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = np.full((T, REPLAY_SLOTS), -1, dtype=np.int32)
    y = np.empty(T, dtype=np.int32)
    V = part.vocab_real
    for t in range(T):
        c = min(int(rng.integers(1, max_ids + 1)), V)
        excluded = None
        if part.n_shards > 1 and rng.random() < empty_shard_frac:
            k = int(rng.integers(0, part.n_shards))
            lo, hi = min(part.ranges[k][0], V), min(part.ranges[k][1], V)
            if V - (hi - lo) > 0:          # never exclude every real id
                excluded = part.ranges[k]
        # the nucleus is ranks 1..c of the Zipf ranking; which vocabulary ids those
        # ranks are is the per-row random permutation drawn here
        if excluded is None:
            chosen = rng.choice(V, size=c, replace=False)
        else:
            lo, hi = excluded
            lo, hi = min(lo, V), min(hi, V)
            pool = V - (hi - lo)
            c = min(c, pool)
            pick = rng.choice(pool, size=c, replace=False)
            chosen = np.where(pick >= lo, pick + (hi - lo), pick)
        n_dup = min(int(round(dup_frac * c)), REPLAY_SLOTS - c)
        dups = rng.choice(chosen, size=n_dup, replace=True) if n_dup else np.empty(0, np.int64)
        slots = np.concatenate([chosen, dups]).astype(np.int32)
        rng.shuffle(slots)
        ids[t, :slots.size] = slots
        y[t] = int(chosen[int(rng.integers(0, c))])
    return ids, y


def upstream_grad(T: int, seed: int = 0) -> np.ndarray:
    """Per-row upstream gradient of the loss with respect to logp, g ~ N(0,1), float32 [T]."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return rng.standard_normal(T, dtype=np.float32)


# ------------------------------------------------------------------ on-device draws
# Same distributions as above, drawn with a seeded torch generator directly on the
# GPU. Used for the large timing inputs of the benchmark, where drawing gigabytes
# on the host would dominate the run; parity tests use the numpy generators above.

def device_forward_inputs(T: int, H: int, part: Partition, tau: float, device, seed: int = 0,
                          w_std: float = 0.02, bias_std: Optional[float] = None):
    """(X bf16 [T,H], [W_k bf16 [V_k,H]], bias list or None, y int32 [T]) on `device`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    X = torch.randn((T, H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = []
    for s, e in part.ranges:
        w = torch.empty((e - s, H), device=device, dtype=torch.bfloat16)
        for r0 in range(0, e - s, 16384):
            r1 = min(e - s, r0 + 16384)
            w[r0:r1] = (torch.randn((r1 - r0, H), generator=g, device=device) * w_std).to(torch.bfloat16)
        W.append(w)
    bias = None
    if bias_std is not None:
        bias = [(torch.randn(e - s, generator=g, device=device) * bias_std).to(torch.bfloat16)
                for s, e in part.ranges]
    y = torch.randint(0, part.vocab_real, (T,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    return X, W, bias, y


def device_logits(T: int, part: Partition, device, seed: int = 0, std: float = 3.0,
                  peak_frac: float = 0.01, peak_value: float = 8.0):
    """Per-shard unscaled bf16 logits [T, V_k] on `device` (peaked rows as in logits_inputs)
    and targets y int32 [T]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    V = part.vocab_padded
    full = torch.empty((T, V), device=device, dtype=torch.bfloat16)
    for r0 in range(0, T, 1024):
        r1 = min(T, r0 + 1024)
        full[r0:r1] = (torch.randn((r1 - r0, V), generator=g, device=device) * std).to(torch.bfloat16)
    n_peak = int(round(peak_frac * part.vocab_real))
    if n_peak:
        for r0 in range(0, T, 1024):
            r1 = min(T, r0 + 1024)
            keys = torch.rand((r1 - r0, part.vocab_real), generator=g, device=device)
            cols = keys.topk(n_peak, dim=1).indices          # uniform without replacement
            full[r0:r1].scatter_(1, cols, torch.full_like(cols, 0, dtype=torch.bfloat16) + peak_value)
    y = torch.randint(0, part.vocab_real, (T,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    return [full[:, s:e] for s, e in part.ranges], y
