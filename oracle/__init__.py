"""fp64 CPU oracle for the deterministic linear-logp operator.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package. The
product path (``lm_head_linear_tcgen05_gb300``) never imports, calls or links
anything here, and this package shares no code with it: it decodes bf16 itself,
does all arithmetic in float64 with numpy, and follows the plain definitions
written out below.

Sources (page title, section):

* "feat(rl-kernel): add CUDA linear logp provider integration", Motivation and
  Changes / Megatron integration: the provider returns selected-token log
  probabilities and optional entropy from output-layer hidden states, the local
  projection weight and bias, the tensor-parallel vocabulary range and the
  real/padded vocabulary sizes; logits may be reused instead of a second
  projection. Tensor parallelism is the vocabulary reduction group.
* "feat(rl-kernel): add ROCm linear logp provider integration", Changes:
  temperature scaling is applied exactly once.
* "Perf/cuda compact top p replay", Summary and Walkthrough ("CUDA kernel and
  empty-shard handling"): the compact replay path sorts and deduplicates up to
  64 ids, applies temperature and returns the local target logit and LSE; an
  empty vocabulary shard gives zero probabilities, LSE = -inf, target logit 0
  and logp = -inf; shard results are reduced in rank order.

Readings where the pages are silent (each one is also listed in the design notes):

* z = (X W^T + b) / tau over the *real* vocabulary; ids >= vocab_real are padding
  and take no part in the softmax.
* logp = z[y] - LSE, LSE = log sum_v exp z_v, entropy = LSE - sum_v p_v z_v (nats).
* Logits given to the logits-reuse path are unscaled (X W^T + b); tau is applied
  once, here.
* Replay ids are 64 int32 slots per row, -1 marks an unused slot; the set R is
  the sorted distinct ids; LSE is taken over R only; logp = -inf if y is not in R.
* Backward is the gradient of sum_t g_t * logp_t, plus sum_t h_t * entropy_t when an
  entropy gradient h is given: G[t,v] = (g_t (1[v = y_t] - p_tv) - h_t p_tv (z_tv -
  mu_t)) / tau with mu_t = sum_v p_tv z_tv; dX = G W, dW = G^T X, db = sum_t G.
* The logits-gather replay scores the replay set from reused unscaled logits
  (z_v = L[t, v] / tau) instead of x . W[v]; everything else as the replay.
* What a shard reports for the rank-ordered reduction: its local LSE, its target
  logit and its own entropy. A replay target inside a non-empty shard's range but
  outside the replay set is an excluded id, whose logit is -inf (page "Perf/cuda
  compact top p replay", Walkthrough: the keep-mask route applies -inf to excluded
  entries); an empty shard keeps the page's target logit 0 and its LSE of -inf
  makes the row's logp -inf when the target falls in it.

Pins (tests/test_oracle.py, CPU only): closed forms (W = 0, constant bias,
two-level logits, one dominant logit), torch.log_softmax in float64 on random
inputs, a pure-Python math.fsum brute force with its own bf16 decode on tiny
inputs, sharded == unsharded, replay with the whole vocabulary as candidate set
== dense LSE, permutation/duplicate invariance, central finite differences of
the backward. Every function below is pinned by at least one of them.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

_W_CHUNK_ROWS = 8192  # decode W to float64 in row chunks to bound host memory


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> float64: the bf16 bits are the high half of an IEEE float32."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- logits

def logits_f64(Xd: np.ndarray, Wd: Sequence[np.ndarray], bd: Optional[Sequence[np.ndarray]],
               ranges, vocab_real: int, tau: float) -> np.ndarray:
    """z[t, v] = (sum_h X[t,h] W_k[v - vs_k, h] + b_k[v - vs_k]) / tau for every real id v.

    Xd [T,H] float64; Wd[k] [V_k,H] float64; bd[k] [V_k] float64 or None.
    Returns float64 [T, vocab_real] in global id order.
    """
    T = Xd.shape[0]
    z = np.empty((T, vocab_real), dtype=np.float64)
    for k, (vs, ve) in enumerate(ranges):
        hi = min(ve, vocab_real)
        if hi <= vs:
            continue
        a = Xd @ Wd[k][: hi - vs].T
        if bd is not None:
            a = a + bd[k][: hi - vs][None, :]
        z[:, vs:hi] = a / tau
    return z


def logits_from_bits(X_bits, W_bits, b_bits, part, tau: float, rows=None) -> np.ndarray:
    """``logits_f64`` on bf16 inputs; ``rows`` selects a subset of rows of X.

    W is decoded chunk by chunk so that full-size LM heads fit in host memory.
    """
    Xd = bf16_to_f64(X_bits if rows is None else X_bits[np.asarray(rows)])
    T = Xd.shape[0]
    z = np.empty((T, part.vocab_real), dtype=np.float64)
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        for c0 in range(0, max(hi - vs, 0), _W_CHUNK_ROWS):
            c1 = min(hi - vs, c0 + _W_CHUNK_ROWS)
            a = Xd @ bf16_to_f64(W_bits[k][c0:c1]).T
            if b_bits is not None:
                a = a + bf16_to_f64(b_bits[k][c0:c1])[None, :]
            z[:, vs + c0: vs + c1] = a / tau
    return z


# ---------------------------------------------------------------------- statistics

def dense_stats(z: np.ndarray, y: np.ndarray):
    """Per row over all columns of z: LSE, logp = z[y] - LSE, entropy = LSE - sum p z.

    Returns float64 arrays (logp, lse, entropy), each [T].
    """
    M = z.max(axis=1)
    S = np.exp(z - M[:, None]).sum(axis=1)
    lse = M + np.log(S)
    p = np.exp(z - lse[:, None])
    entropy = lse - (p * z).sum(axis=1)
    logp = z[np.arange(z.shape[0]), y] - lse
    return logp, lse, entropy


@dataclass
class ShardStats:
    """Local statistics of one vocabulary shard, per row.

    lse: log sum over the shard's real ids of exp z (-inf if the shard has none);
    h:   the shard's own entropy, lse - sum over those ids of softmax_local(z) * z
         (0 if the shard is empty);
    t:   z[y] if y lies in the shard, else 0.
    """
    lse: np.ndarray
    h: np.ndarray
    t: np.ndarray


def shard_stats(z: np.ndarray, y: np.ndarray, ranges, vocab_real: int) -> List[ShardStats]:
    """Local statistics of each shard (empty shard: lse = -inf, h = 0, t = 0)."""
    T = z.shape[0]
    out = []
    for vs, ve in ranges:
        hi = min(ve, vocab_real)
        in_shard = (y >= vs) & (y < ve)
        t = np.where(in_shard, z[np.arange(T), np.clip(y, 0, vocab_real - 1)], 0.0)
        if hi <= vs:
            out.append(ShardStats(np.full(T, -np.inf), np.zeros(T), t))
            continue
        zk = z[:, vs:hi]
        M = zk.max(axis=1)
        S = np.exp(zk - M[:, None]).sum(axis=1)
        lse = M + np.log(S)
        h = lse - (np.exp(zk - lse[:, None]) * zk).sum(axis=1)
        out.append(ShardStats(lse, h, t))
    return out


def merge_shard_stats(lse: np.ndarray, t: np.ndarray, h: np.ndarray, y: np.ndarray, ranges, vocab_real: int):
    """Combine per-shard statistics [K, T] of the shards `ranges` (ascending, the
    rank-ordered reduction) into per-row (logp, lse, entropy).

    LSE = log sum_k exp(lse_k) (an empty shard, lse_k = -inf, adds nothing);
    entropy = -sum_v p_v log p_v = sum_k w_k (h_k + LSE - lse_k) with w_k = exp(lse_k - LSE),
    the share of shard k in the softmax; logp = t_o - LSE where o is the shard holding y,
    and -inf when no shard holds y, when that shard is empty (the page's empty-shard rule)
    or when its target logit is -inf (an excluded id). A row whose shards are all empty
    gets LSE = -inf, logp = -inf, entropy = 0.
    """
    lse = np.asarray(lse, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    K, T = lse.shape
    M = lse.max(axis=0)
    out_lse = np.full(T, -np.inf)
    ent = np.zeros(T)
    logp = np.full(T, -np.inf)
    live = np.isfinite(M)
    Ml = M[live]
    acc = np.zeros(Ml.shape)
    for k in range(K):                                   # ascending shard order
        l = lse[k, live]
        acc += np.where(np.isfinite(l), np.exp(np.where(np.isfinite(l), l, 0.0) - Ml), 0.0)
    out_lse[live] = Ml + np.log(acc)
    L = out_lse[live]
    for k in range(K):
        l = lse[k, live]
        fin = np.isfinite(l)
        w = np.where(fin, np.exp(np.where(fin, l, 0.0) - L), 0.0)
        ent[live] += w * (h[k, live] + np.where(fin, L - np.where(fin, l, 0.0), 0.0))
    for k, (vs, ve) in enumerate(ranges):
        own = live & (y >= vs) & (y < ve) & (y < vocab_real) & np.isfinite(lse[k])
        logp[own] = t[k, own] - out_lse[own]
    return logp, out_lse, ent


def merge_shards(stats: List[ShardStats], y: np.ndarray, ranges, vocab_real: Optional[int] = None):
    """``merge_shard_stats`` on a list of ShardStats (ascending shard order)."""
    vr = int(ranges[-1][1]) if vocab_real is None else vocab_real
    return merge_shard_stats(np.stack([s.lse for s in stats]), np.stack([s.t for s in stats]),
                             np.stack([s.h for s in stats]), y, ranges, vr)


# ------------------------------------------------------------------------- forward

@dataclass
class ForwardResult:
    logp: np.ndarray
    lse: np.ndarray
    entropy: np.ndarray
    shards: List[ShardStats]


def forward(X_bits, W_bits, b_bits, part, y, tau: float, rows=None) -> ForwardResult:
    """Fused linear-logp forward on bf16 inputs (optionally on a subset of rows)."""
    yy = np.asarray(y if rows is None else np.asarray(y)[np.asarray(rows)], dtype=np.int64)
    z = logits_from_bits(X_bits, W_bits, b_bits, part, tau, rows)
    logp, lse, ent = dense_stats(z, yy)
    return ForwardResult(logp, lse, ent, shard_stats(z, yy, part.ranges, part.vocab_real))


def forward_from_logits(L_bits, part, y, tau: float, rows=None) -> ForwardResult:
    """Logits-reuse forward: L_bits[k] are the unscaled bf16 logits [T, V_k] of shard k.

    z = L / tau (temperature applied once, here) over the real ids.
    """
    sel = slice(None) if rows is None else np.asarray(rows)
    yy = np.asarray(y, dtype=np.int64)[sel]
    T = yy.shape[0]
    z = np.empty((T, part.vocab_real), dtype=np.float64)
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        if hi > vs:
            z[:, vs:hi] = bf16_to_f64(L_bits[k][sel][:, : hi - vs]) / tau
    logp, lse, ent = dense_stats(z, yy)
    return ForwardResult(logp, lse, ent, shard_stats(z, yy, part.ranges, part.vocab_real))


# -------------------------------------------------------------------------- replay

def replay_set(slots: np.ndarray, vocab_real: int) -> np.ndarray:
    """Sorted distinct ids of one row's replay slots; -1 marks an unused slot."""
    s = np.asarray(slots, dtype=np.int64)
    s = s[s != -1]
    if np.any((s < 0) | (s >= vocab_real)):
        raise ValueError("replay id outside [0, vocab_real)")
    return np.unique(s)


@dataclass
class ReplayResult:
    logp: np.ndarray
    lse: np.ndarray
    shard_lse: np.ndarray   # [K, T]
    shard_t: np.ndarray     # [K, T]


def top_p_replay(X_bits, W_bits, b_bits, part, ids, y, tau: float, rows=None) -> ReplayResult:
    """Compact top-p replay: LSE and target logp over each row's replay set only.

    For row t with set R (sorted, distinct): z_v = (x_t . W[v] + b[v]) / tau for
    v in R; LSE_R = log sum_{v in R} exp z_v; logp = z_y - LSE_R if y in R else
    -inf. Per shard k: the same over R restricted to the shard, with the empty
    shard convention (lse -inf, t 0) when that restriction is empty; a target that lies
    in a non-empty shard's range but not in R is an excluded id, whose logit the
    keep-mask route sets to -inf, so that shard's t is -inf.
    """
    rows = np.arange(np.asarray(ids).shape[0]) if rows is None else np.asarray(rows)
    K = part.n_shards
    T = rows.shape[0]
    logp = np.full(T, -np.inf)
    lse = np.full(T, -np.inf)
    sh_lse = np.full((K, T), -np.inf)
    sh_t = np.zeros((K, T))
    starts = np.array([r[0] for r in part.ranges])
    for i, r in enumerate(rows):
        R = replay_set(ids[r], part.vocab_real)
        if R.size == 0:
            continue
        x = bf16_to_f64(X_bits[r])
        zs = np.empty(R.size)
        for j, v in enumerate(R):
            k = int(np.searchsorted(starts, v, side="right") - 1)
            vs = part.ranges[k][0]
            a = float(np.dot(x, bf16_to_f64(W_bits[k][v - vs])))
            if b_bits is not None:
                a += float(bf16_to_f64(b_bits[k][v - vs: v - vs + 1])[0])
            zs[j] = a / tau
        M = zs.max()
        lse[i] = M + np.log(np.exp(zs - M).sum())
        yi = int(y[r])
        hit = np.nonzero(R == yi)[0]
        if hit.size:
            logp[i] = zs[hit[0]] - lse[i]
        for k, (vs, ve) in enumerate(part.ranges):
            m = (R >= vs) & (R < ve)
            if not m.any():
                continue
            zk = zs[m]
            Mk = zk.max()
            sh_lse[k, i] = Mk + np.log(np.exp(zk - Mk).sum())
            if vs <= yi < ve:
                sh_t[k, i] = zs[hit[0]] if hit.size else -np.inf
    return ReplayResult(logp, lse, sh_lse, sh_t)


def top_p_replay_from_logits(L_bits, part, ids, y, tau: float, rows=None) -> ReplayResult:
    """Compact top-p replay scored from reused local logits: z_v = L_k[t, v - vs_k] / tau
    for v in the row's sorted distinct set R (temperature once, here); LSE over R;
    logp = z_y - LSE_R if y in R else -inf; per-shard local LSE and target logit with
    the empty-shard convention. Same set rules as ``top_p_replay``."""
    rows = np.arange(np.asarray(ids).shape[0]) if rows is None else np.asarray(rows)
    K = part.n_shards
    T = rows.shape[0]
    logp = np.full(T, -np.inf)
    lse = np.full(T, -np.inf)
    sh_lse = np.full((K, T), -np.inf)
    sh_t = np.zeros((K, T))
    starts = np.array([r[0] for r in part.ranges])
    for i, r in enumerate(rows):
        R = replay_set(ids[r], part.vocab_real)
        if R.size == 0:
            continue
        zs = np.empty(R.size)
        for j, v in enumerate(R):
            k = int(np.searchsorted(starts, v, side="right") - 1)
            zs[j] = float(bf16_to_f64(L_bits[k][r, v - part.ranges[k][0]: v - part.ranges[k][0] + 1])[0]) / tau
        M = zs.max()
        lse[i] = M + np.log(np.exp(zs - M).sum())
        yi = int(y[r])
        hit = np.nonzero(R == yi)[0]
        if hit.size:
            logp[i] = zs[hit[0]] - lse[i]
        for k, (vs, ve) in enumerate(part.ranges):
            m = (R >= vs) & (R < ve)
            if not m.any():
                continue
            zk = zs[m]
            Mk = zk.max()
            sh_lse[k, i] = Mk + np.log(np.exp(zk - Mk).sum())
            if vs <= yi < ve:
                sh_t[k, i] = zs[hit[0]] if hit.size else -np.inf
    return ReplayResult(logp, lse, sh_lse, sh_t)


# ------------------------------------------------------------------------ backward

@dataclass
class BackwardResult:
    dX: np.ndarray                 # [T, H]
    dW: List[np.ndarray]           # per shard [len(dw_rows_k), H] (all rows by default)
    db: List[np.ndarray]           # per shard [len(dw_rows_k)]
    dw_rows: List[np.ndarray]      # local row indices of each shard that dW/db cover


def backward_f64(Xd, Wd, bd, ranges, vocab_real, y, tau, g, dw_rows=None, h=None) -> BackwardResult:
    """Gradient of sum_t g_t logp_t (+ sum_t h_t entropy_t when h is given) with respect
    to X, W_k and b_k (float64 inputs).

    p = softmax(z) over the real ids, mu_t = sum_v p_tv z_tv;
    G[t,v] = (g_t (1[v = y_t] - p_tv) - h_t p_tv (z_tv - mu_t)) / tau on real ids and 0
    on padded ids (d entropy / d z_v = -p_v (z_v - mu)); dX = sum_k G_k W_k;
    dW_k = G_k^T X; db_k = sum_t G_k.
    """
    y = np.asarray(y, dtype=np.int64)
    z = logits_f64(Xd, Wd, bd, ranges, vocab_real, tau)
    T = z.shape[0]
    M = z.max(axis=1, keepdims=True)
    p = np.exp(z - M)
    p /= p.sum(axis=1, keepdims=True)
    onehot = np.zeros_like(p)
    onehot[np.arange(T), y] = 1.0
    G = np.asarray(g, dtype=np.float64)[:, None] * (onehot - p) / tau   # [T, vocab_real]
    if h is not None:
        mu = (p * z).sum(axis=1, keepdims=True)
        G -= np.asarray(h, dtype=np.float64)[:, None] * p * (z - mu) / tau
    H = Xd.shape[1]
    dX = np.zeros((T, H))
    dW, db, rows_out = [], [], []
    for k, (vs, ve) in enumerate(ranges):
        Vk = ve - vs
        hi = min(ve, vocab_real)
        Gk = np.zeros((T, Vk))
        if hi > vs:
            Gk[:, : hi - vs] = G[:, vs:hi]
        dX += Gk @ Wd[k]
        rk = np.arange(Vk) if dw_rows is None else np.asarray(dw_rows[k], dtype=np.int64)
        dW.append(Gk[:, rk].T @ Xd)
        db.append(Gk[:, rk].sum(axis=0))
        rows_out.append(rk)
    return BackwardResult(dX, dW, db, rows_out)


def backward(X_bits, W_bits, b_bits, part, y, tau, g, dw_rows=None, h=None) -> BackwardResult:
    """``backward_f64`` on bf16 inputs. ``dw_rows[k]`` (local indices) limits dW/db to a
    sample; ``h`` is the optional upstream gradient of the entropy."""
    Xd = bf16_to_f64(X_bits)
    Wd = [bf16_to_f64(w) for w in W_bits]
    bd = None if b_bits is None else [bf16_to_f64(b) for b in b_bits]
    return backward_f64(Xd, Wd, bd, part.ranges, part.vocab_real, y, tau, g, dw_rows, h)


def backward_sampled(X_bits, W_bits, b_bits, part, y, tau, g, dx_rows, dw_rows):
    """Backward at full size on samples: dX on rows ``dx_rows`` (each needs only its own
    row of z) and dW/db on local vocab rows ``dw_rows[k]`` (each needs the full
    column of G, hence every row's LSE, computed here chunk by chunk over W).

    Returns (dX [len(dx_rows), H], [dW_k sample], [db_k sample]).
    """
    y = np.asarray(y, dtype=np.int64)
    g = np.asarray(g, dtype=np.float64)
    T = X_bits.shape[0]
    Xd = bf16_to_f64(X_bits)
    # LSE of the rows needed: every row when dW/db samples are asked for (a column
    # of G spans all rows), else only the dX rows. Streamed over W chunks with an
    # online max / sum in float64.
    need = np.arange(T) if any(len(r) for r in dw_rows) else np.asarray(dx_rows)
    M = np.full(need.size, -np.inf)
    S = np.zeros(need.size)
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        for c0 in range(0, max(hi - vs, 0), _W_CHUNK_ROWS):
            c1 = min(hi - vs, c0 + _W_CHUNK_ROWS)
            a = Xd[need] @ bf16_to_f64(W_bits[k][c0:c1]).T
            if b_bits is not None:
                a = a + bf16_to_f64(b_bits[k][c0:c1])[None, :]
            z = a / tau
            Mn = np.maximum(M, z.max(axis=1))
            S = S * np.exp(M - Mn) + np.exp(z - Mn[:, None]).sum(axis=1)
            M = Mn
    lse = np.full(T, np.nan)
    lse[need] = M + np.log(S)
    # dX on the sampled rows: G_row = g (onehot - p)/tau, dX = G_row W
    dx_rows = np.asarray(dx_rows)
    H = X_bits.shape[1]
    dX = np.zeros((dx_rows.size, H))
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        for c0 in range(0, max(hi - vs, 0), _W_CHUNK_ROWS):
            c1 = min(hi - vs, c0 + _W_CHUNK_ROWS)
            Wc = bf16_to_f64(W_bits[k][c0:c1])
            a = Xd[dx_rows] @ Wc.T
            if b_bits is not None:
                a = a + bf16_to_f64(b_bits[k][c0:c1])[None, :]
            z = a / tau
            G = -np.exp(z - lse[dx_rows][:, None])
            ids = np.arange(vs + c0, vs + c1)
            G = G + (y[dx_rows][:, None] == ids[None, :])
            G *= (g[dx_rows] / tau)[:, None]
            dX += G @ Wc
    dW, db = [], []
    for k, (vs, ve) in enumerate(part.ranges):
        rk = np.asarray(dw_rows[k], dtype=np.int64)
        if rk.size == 0:
            dW.append(np.zeros((0, H)))
            db.append(np.zeros(0))
            continue
        Wr = bf16_to_f64(W_bits[k][rk])
        a = Xd @ Wr.T
        if b_bits is not None:
            a = a + bf16_to_f64(b_bits[k][rk])[None, :]
        z = a / tau
        gid = vs + rk
        G = (y[:, None] == gid[None, :]) - np.exp(z - lse[:, None])
        G *= (g / tau)[:, None]
        G[:, gid >= part.vocab_real] = 0.0
        dW.append(G.T @ Xd)
        db.append(G.sum(axis=0))
    return dX, dW, db


def backward_from_logits(L_bits, part, y, tau, g, h=None, rows=None) -> List[np.ndarray]:
    """Gradient of sum_t g_t logp_t (+ sum_t h_t entropy_t) of ``forward_from_logits`` with
    respect to the reused unscaled logits L_k (the route that avoids a second projection).

    z = L / tau, so dL = G with G[t,v] = (g_t (1[v = y_t] - p_tv) - h_t p_tv (z_tv - mu_t)) / tau
    on real ids and 0 on padded ids, exactly the G of ``backward_f64``. Returns one float64
    [T, V_k] array per shard (``rows`` selects rows of L, y, g and h).
    """
    sel = slice(None) if rows is None else np.asarray(rows)
    yy = np.asarray(y, dtype=np.int64)[sel]
    gg = np.asarray(g, dtype=np.float64)[sel]
    T = yy.shape[0]
    z = np.empty((T, part.vocab_real), dtype=np.float64)
    for k, (vs, ve) in enumerate(part.ranges):
        hi = min(ve, part.vocab_real)
        if hi > vs:
            z[:, vs:hi] = bf16_to_f64(L_bits[k][sel][:, : hi - vs]) / tau
    M = z.max(axis=1, keepdims=True)
    p = np.exp(z - M)
    p /= p.sum(axis=1, keepdims=True)
    G = -p
    G[np.arange(T), yy] += 1.0
    G *= (gg / tau)[:, None]
    if h is not None:
        hh = np.asarray(h, dtype=np.float64)[sel]
        mu = (p * z).sum(axis=1, keepdims=True)
        G -= (hh / tau)[:, None] * p * (z - mu)
    out = []
    for k, (vs, ve) in enumerate(part.ranges):
        dL = np.zeros((T, ve - vs))
        hi = min(ve, part.vocab_real)
        if hi > vs:
            dL[:, : hi - vs] = G[:, vs:hi]
        out.append(dL)
    return out
