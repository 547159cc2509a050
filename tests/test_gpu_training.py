"""GPU parity of the training-side entry points against the fp64 oracle:

* lp_backward_from_logits (gradient with respect to reused logits): bf16 and fp32
  outputs, in place, ragged widths, padded ids, empty shards, the entropy term, rows
  with no gradient; full size (T=8192 x 151936) on sampled rows;
* lp_backward_ex: bf16 dX is the fp32 dX rounded once (bitwise), for one K range and for
  several; accumulation into caller dW / db is one fp32 add per element (bitwise);
* the autograd wrappers: gradients equal the library calls bit for bit and match the
  oracle within tolerance.
"""
import numpy as np
import pytest

import oracle
import synth
from lp_util import TOL_GRAD_REL, dev_bf16, dev_f32, dev_i32, dev_inputs, part_of, rel_fro

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
    import torch
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def _dev_logits(L):
    """Shard logits on the device as [T, V_k] views of buffers whose row stride is V_k
    rounded up to 8 (the 16-byte row rule); None for empty shards."""
    import torch
    out = []
    for a in L:
        T, w = a.shape
        if w == 0:
            out.append(None)
            continue
        buf = torch.zeros((T, (w + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")
        buf[:, :w] = dev_bf16(a)
        out.append(buf[:, :w])
    return out


def _check_grad(got, ref, ctx):
    """Per shard: relative Frobenius error within the gradient tolerance and every
    element within 1 % of the shard's largest reference entry."""
    for k, (g, r) in enumerate(zip(got, ref)):
        if r.shape[1] == 0:
            assert g is None, (ctx, k)
            continue
        a = _np(g).astype(np.float64)
        assert a.shape == r.shape, (ctx, k)
        assert rel_fro(a, r) <= TOL_GRAD_REL, (ctx, k, rel_fro(a, r))
        scale = max(float(np.abs(r).max()), 1e-30)
        assert float(np.abs(a - r).max()) <= 1e-2 * scale, (ctx, k)


# -------------------------------------------------------- gradient w.r.t. logits

CASES = [
    (37, [0, 1000], 1000, 0.7),
    (64, [0, 4099, 4099, 9000, 12301], 12290, 1.3),   # ragged widths, empty shard, padding
    (5, [0, 7], 7, 0.3),                                 # narrower than one vector
    (130, [0, 2048, 4096, 6144, 8192], 8000, 2.5),      # a shard of padding only at the end
]


@pytest.mark.parametrize("T,bounds,real,tau", CASES)
@pytest.mark.parametrize("entropy_term", [False, True])
def test_logits_backward_parity(lp, T, bounds, real, tau, entropy_term):
    import torch
    part = synth.ranges_partition(real, bounds[-1], bounds)
    L, y, tau = synth.logits_inputs(T, part, tau, seed=T + 3)
    g = synth.upstream_grad(T, seed=T)
    h = synth.upstream_grad(T, seed=T + 1) if entropy_term else None
    Ld = _dev_logits(L)
    P = part_of(part)
    fwd = lp.lp_forward_from_logits(Ld, P, dev_i32(y), tau)
    ent = fwd["entropy"] if entropy_term else None
    hd = dev_f32(h) if entropy_term else None
    ref = oracle.backward_from_logits(L, part, y, tau, g, h=h)
    ctx = f"T={T} bounds={bounds} real={real} tau={tau} h={entropy_term}"
    for dt in (torch.bfloat16, torch.float32):
        dL = lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], dev_f32(g), entropy=ent,
                                        grad_entropy=hd, out_dtype=dt)
        assert lp.lp_get_device_error() == 0, ctx
        _check_grad(dL, ref, (ctx, dt))
        for d, (s, e) in zip(dL, part.ranges):            # padded ids: exactly zero
            if d is not None and e > real:
                assert torch.all(d[:, max(real - s, 0):] == 0), ctx
        if dt == torch.float32:
            d32 = dL
        else:
            d16 = dL
    # bf16 output is the fp32 output rounded once
    for a, b in zip(d16, d32):
        if a is not None:
            assert torch.equal(a, b.to(torch.bfloat16)), ctx
    # in place over the logits: same bits as out of place
    Lin = _dev_logits(L)
    got = lp.lp_backward_from_logits(Lin, P, dev_i32(y), tau, fwd["lse"], dev_f32(g), entropy=ent,
                                     grad_entropy=hd, out=Lin)
    for a, b in zip(got, d16):
        if b is not None:
            assert torch.equal(a, b), ctx
    # run to run and batch invariant: a slice of rows gives the same bits
    again = lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], dev_f32(g), entropy=ent,
                                       grad_entropy=hd)
    for a, b in zip(again, d16):
        if b is not None:
            assert torch.equal(a, b), ctx
    if T > 3:
        r0, r1 = 1, T - 1
        sub = lp.lp_backward_from_logits([None if x is None else x[r0:r1] for x in Ld], P,
                                         dev_i32(y[r0:r1]), tau, fwd["lse"][r0:r1].contiguous(),
                                         dev_f32(g[r0:r1]), entropy=None if ent is None else ent[r0:r1].contiguous(),
                                         grad_entropy=None if hd is None else hd[r0:r1].contiguous())
        for a, b in zip(sub, d16):
            if b is not None:
                assert torch.equal(a, b[r0:r1]), ctx


def test_logits_backward_rows_without_gradient_are_zero(lp):
    import torch
    part = synth.ranges_partition(900, 904, [0, 452, 904])
    T = 6
    L, y, tau = synth.logits_inputs(T, part, 0.7, seed=40)
    Ld = _dev_logits(L)
    P = part_of(part)
    fwd = lp.lp_forward_from_logits(Ld, P, dev_i32(y), tau)
    lse = fwd["lse"].clone()
    g = torch.ones(T, dtype=torch.float32, device="cuda")
    lse[1] = float("inf")
    lse[2] = float("nan")
    g[3] = float("inf")
    g[4] = 0.0
    dL = lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, lse, g, out_dtype=torch.float32)
    full = torch.cat([d for d in dL], dim=1)
    assert not torch.isnan(full).any()
    for r in (1, 2, 3, 4):
        assert torch.all(full[r] == 0), r
    assert torch.any(full[0] != 0) and torch.any(full[5] != 0)
    # -inf logits (entries masked out by the caller) get zero gradient, also with the entropy term
    Lm = _dev_logits(L)
    col = 5 if int(y[0]) != 5 else 6
    Lm[0][0, col] = float("-inf")
    fm = lp.lp_forward_from_logits(Lm, P, dev_i32(y), tau)
    dm = lp.lp_backward_from_logits(Lm, P, dev_i32(y), tau, fm["lse"], torch.ones(T, device="cuda"),
                                    entropy=fm["entropy"], grad_entropy=torch.ones(T, device="cuda"),
                                    out_dtype=torch.float32)
    assert dm[0][0, col].item() == 0.0 and not torch.isnan(dm[0]).any() and not torch.isnan(dm[1]).any()


def test_logits_backward_rejects_bad_arguments(lp):
    import torch
    part = synth.ranges_partition(96, 96, [0, 48, 96])
    T = 4
    L, y, tau = synth.logits_inputs(T, part, 0.7, seed=41)
    Ld = _dev_logits(L)
    P = part_of(part)
    fwd = lp.lp_forward_from_logits(Ld, P, dev_i32(y), tau)
    g = torch.ones(T, dtype=torch.float32, device="cuda")
    # shard 0's output overlapping shard 1's logits
    other = torch.empty((T, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lp.LPError, match="INVALID_ARG"):
        lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], g, out=[Ld[1], other])
    # an fp32 output that starts 4 bytes past a 16-byte boundary
    wide = torch.empty((T, 52), dtype=torch.float32, device="cuda")
    with pytest.raises(lp.LPError, match="ALIGNMENT"):
        lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], g, out_dtype=torch.float32,
                                   out=[wide[:, 1:49], torch.empty((T, 48), dtype=torch.float32, device="cuda")])
    with pytest.raises(ValueError):
        lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], g, entropy=fwd["entropy"])


def test_logits_backward_full_size_sampled_rows(lp):
    # the logits-reuse workload: T=8192 x 151936 bf16 logits, 1 % peaked entries per row
    import torch
    part = synth.even_partition(151936, 1)
    T = 8192
    L, y, tau = synth.logits_inputs(T, part, 0.7, seed=42)
    g = synth.upstream_grad(T, seed=42)
    h = synth.upstream_grad(T, seed=43)
    Ld = [dev_bf16(L[0])]
    P = part_of(part)
    fwd = lp.lp_forward_from_logits(Ld, P, dev_i32(y), tau)
    dL = lp.lp_backward_from_logits(Ld, P, dev_i32(y), tau, fwd["lse"], dev_f32(g), entropy=fwd["entropy"],
                                    grad_entropy=dev_f32(h))
    assert lp.lp_get_device_error() == 0
    rows = np.unique(np.concatenate([[0, 1, T // 2, T - 1], np.random.default_rng(44).choice(T, 60, replace=False)]))
    ref = oracle.backward_from_logits(L, part, y, tau, g, h=h, rows=rows)
    _check_grad([dL[0][torch.as_tensor(rows, device="cuda")]], ref, "full size")
    # every row sums to ~0 (sum_v (1[v=y] - p_v) = 0 and sum_v p_v (z_v - mu) = 0)
    rs = dL[0].float().sum(dim=1).abs().max().item()
    assert rs <= 1e-2 * float(np.abs(g).max() + np.abs(h).max() * 10) / tau


# ----------------------------------------------------- lp_backward_ex options

@pytest.mark.parametrize("V,bounds", [
    (3000, [0, 1500, 3008]),                 # one K range: dX rounded in the GEMM epilogue
    (70000, [0, 35000, 70016]),              # two K ranges: dX rounded in the ordered reduction
])
def test_backward_ex_bf16_dx_and_accumulate(lp, V, bounds):
    import torch
    part = synth.ranges_partition(V, bounds[-1], bounds)
    T, H = 200, 136
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=V % 97, w_std=0.5 / np.sqrt(H), bias_std=0.05)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    g = dev_f32(synth.upstream_grad(T, seed=5))
    fwd = lp.lp_forward(X, W, b, P, y, inp.tau)
    base = lp.lp_backward(X, W, b, P, y, inp.tau, fwd["lse"], g)
    ex = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], g, dx_dtype=torch.bfloat16)
    assert lp.lp_get_device_error() == 0
    assert ex["dX"].dtype == torch.bfloat16
    assert torch.equal(ex["dX"], base["dX"].to(torch.bfloat16))
    for k in range(len(bounds) - 1):
        assert torch.equal(ex["dW"][k], base["dW"][k]) and torch.equal(ex["db"][k], base["db"][k])
    # bf16 dW: the same fp32 result rounded once; padded ids exactly zero
    e16 = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], g, dw_dtype=torch.bfloat16)
    for k, (s, e) in enumerate(part.ranges):
        assert e16["dW"][k].dtype == torch.bfloat16
        assert torch.equal(e16["dW"][k], base["dW"][k].to(torch.bfloat16)), k
        assert torch.equal(e16["db"][k], base["db"][k]), k
        real = max(min(e, V) - s, 0)
        assert torch.all(e16["dW"][k][real:] == 0), k
    assert torch.equal(e16["dX"], base["dX"])
    # accumulate: one fp32 add onto the caller's buffers; padded ids keep their values
    gen = torch.Generator(device="cuda").manual_seed(7)
    dW0 = [torch.randn(w.shape, generator=gen, device="cuda") for w in base["dW"]]
    db0 = [torch.randn(d.shape, generator=gen, device="cuda") for d in base["db"]]
    acc = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], g, accumulate=True,
                            dW=[t.clone() for t in dW0], db=[t.clone() for t in db0])
    for k, (s, e) in enumerate(part.ranges):
        real = max(min(e, V) - s, 0)
        assert torch.equal(acc["dW"][k][:real], dW0[k][:real] + base["dW"][k][:real]), k
        assert torch.equal(acc["db"][k][:real], db0[k][:real] + base["db"][k][:real]), k
        assert torch.equal(acc["dW"][k][real:], dW0[k][real:]) and torch.equal(acc["db"][k][real:], db0[k][real:])
    assert torch.equal(acc["dX"], base["dX"])
    # with the entropy term too, against the oracle
    h = synth.upstream_grad(T, seed=6)
    exh = lp.lp_backward_ex(X, W, b, P, y, inp.tau, fwd["lse"], g, entropy=fwd["entropy"], grad_entropy=dev_f32(h),
                            dx_dtype=torch.bfloat16)
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, _np(g), h=h)
    assert rel_fro(_np(exh["dX"]), ref.dX) <= TOL_GRAD_REL
    for k in range(len(bounds) - 1):
        assert rel_fro(_np(exh["dW"][k]), ref.dW[k]) <= TOL_GRAD_REL
    # an empty batch leaves accumulated buffers untouched
    keep = [t.clone() for t in dW0]
    lp.lp_backward_ex(X[:0], W, b, P, y[:0], inp.tau, fwd["lse"][:0], g[:0], accumulate=True, dW=keep,
                      db=[t.clone() for t in db0])
    torch.cuda.synchronize()
    assert all(torch.equal(a, c) for a, c in zip(keep, dW0))


def test_backward_ex_rejects_bad_options(lp):
    import torch
    part = synth.ranges_partition(64, 64, [0, 64])
    inp = synth.forward_inputs(4, 16, part, tau=1.0, seed=1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    g = torch.ones(4, device="cuda")
    lse = torch.zeros(4, device="cuda")
    with pytest.raises(TypeError):
        lp.lp_backward_ex(X, W, b, P, y, 1.0, lse, g, dx_dtype=torch.float16)
    with pytest.raises(ValueError):
        lp.lp_backward_ex(X, W, b, P, y, 1.0, lse, g, accumulate=True)
    with pytest.raises(ValueError):
        lp.lp_backward_ex(X, W, b, P, y, 1.0, lse, g, accumulate=True, dw_dtype=torch.bfloat16,
                          dW=[torch.zeros((64, 16), dtype=torch.bfloat16, device="cuda")],
                          db=[torch.zeros(64, device="cuda")])


# ------------------------------------------------------------------- autograd

def test_autograd_fused_route_matches_library_and_oracle(lp):
    import torch
    from lm_head_linear_tcgen05_gb300.autograd import linear_logp
    part = synth.ranges_partition(2000, 2048, [0, 1024, 1024, 2048])      # an empty shard, padding
    T, H = 150, 64
    inp = synth.forward_inputs(T, H, part, tau=0.8, seed=9, w_std=0.5 / np.sqrt(H), bias_std=0.05)
    X0, W0, b0, y = dev_inputs(inp)
    X = X0.clone().requires_grad_(True)
    W = [None if w is None else w.clone().requires_grad_(True) for w in W0]
    b = [None if x is None else x.clone().requires_grad_(True) for x in b0]
    P = part_of(part)
    a = synth.upstream_grad(T, seed=10)
    c = synth.upstream_grad(T, seed=11)
    logp, ent = linear_logp(X, W, b, P, y, inp.tau)
    assert logp.requires_grad and ent.requires_grad
    ((logp * dev_f32(a)).sum() + (ent * dev_f32(c)).sum()).backward()
    # the same bits as the library calls
    fwd = lp.lp_forward(X0, W0, b0, P, y, inp.tau)
    assert torch.equal(logp.detach(), fwd["logp"]) and torch.equal(ent.detach(), fwd["entropy"])
    r = lp.lp_backward_ex(X0, W0, b0, P, y, inp.tau, fwd["lse"], dev_f32(a), entropy=fwd["entropy"],
                          grad_entropy=dev_f32(c), dx_dtype=torch.bfloat16)
    assert torch.equal(X.grad, r["dX"])
    for k in (0, 2):
        assert torch.equal(W[k].grad, r["dW"][k].to(torch.bfloat16))
        assert torch.equal(b[k].grad, r["db"][k].to(torch.bfloat16))
    ref = oracle.backward(inp.X, inp.W, inp.bias, part, inp.y, inp.tau, a, h=c)
    assert rel_fro(_np(X.grad), ref.dX) <= TOL_GRAD_REL
    for k in (0, 2):
        assert rel_fro(_np(W[k].grad), ref.dW[k]) <= TOL_GRAD_REL
        assert rel_fro(_np(b[k].grad), ref.db[k]) <= TOL_GRAD_REL
    # logp alone: the entropy output unused
    X.grad = None
    logp, _ = linear_logp(X, W, b, P, y, inp.tau)
    (logp * dev_f32(a)).sum().backward()
    r = lp.lp_backward_ex(X0, W0, b0, P, y, inp.tau, fwd["lse"], dev_f32(a), dx_dtype=torch.bfloat16)
    assert torch.equal(X.grad, r["dX"])


def test_autograd_logits_route_matches_library_and_oracle(lp):
    import torch
    from lm_head_linear_tcgen05_gb300.autograd import linear_logp_from_logits
    part = synth.ranges_partition(5000, 5008, [0, 2504, 5008])   # rows of whole 16-byte vectors
    T = 70
    L, y, tau = synth.logits_inputs(T, part, 0.7, seed=12)
    Ld = [x.clone().requires_grad_(True) for x in _dev_logits(L)]
    P = part_of(part)
    a = synth.upstream_grad(T, seed=13)
    c = synth.upstream_grad(T, seed=14)
    logp, ent = linear_logp_from_logits(Ld, P, dev_i32(y), tau)
    ((logp * dev_f32(a)).sum() + (ent * dev_f32(c)).sum()).backward()
    fwd = lp.lp_forward_from_logits([x.detach() for x in Ld], P, dev_i32(y), tau)
    r = lp.lp_backward_from_logits([x.detach() for x in Ld], P, dev_i32(y), tau, fwd["lse"], dev_f32(a),
                                   entropy=fwd["entropy"], grad_entropy=dev_f32(c))
    ref = oracle.backward_from_logits(L, part, y, tau, a, h=c)
    for k in range(2):
        assert torch.equal(Ld[k].grad, r[k])
    _check_grad([x.grad for x in Ld], ref, "autograd logits")
