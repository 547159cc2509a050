"""torch.autograd wrappers: the provider's outputs with gradients attached.

Page "feat(rl-kernel): add CUDA linear logp provider integration", Summary and
Changes: the provider returns log probabilities and optional entropy, and the
caller rejects detached gradients, so both outputs must carry gradients back to
whatever produced them - the hidden states, projection weight and bias on the fused
route, or the reused logits on the logits-reuse route.

Each forward runs one library call and keeps its merged LSE and entropy for the
backward, which is again one library call (three tcgen05 GEMMs plus reductions on the
fused route, one streaming kernel on the logits route). Nothing here computes: the
wrappers only route tensors between the two calls.

    logp, entropy = linear_logp(X, [W], None, part, y, tau)
    (logp * advantages).sum().backward()       # X.grad, W.grad
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import lp_backward_ex, lp_backward_from_logits, lp_forward, lp_forward_from_logits


def _zeros_like_rows(ref: torch.Tensor) -> torch.Tensor:
    return torch.zeros(ref.shape[0], dtype=torch.float32, device=ref.device)


def _f32(g: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    return None if g is None else g.to(torch.float32).contiguous()


class _LinearLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, part, y, tau, n, has_bias, *wb):
        W = list(wb[:n])
        bias = list(wb[n:]) if has_bias else None
        out = lp_forward(X, W, bias, part, y, tau, entropy=True)
        ctx.part, ctx.tau, ctx.n, ctx.has_bias = part, tau, n, has_bias
        ctx.save_for_backward(X, y, out["lse"], out["entropy"], *wb)
        ctx.mark_non_differentiable(out["lse"])
        ctx.set_materialize_grads(False)
        return out["logp"], out["entropy"], out["lse"]

    @staticmethod
    def backward(ctx, g_logp, g_entropy, _g_lse):
        X, y, lse, entropy, *wb = ctx.saved_tensors
        n = ctx.n
        W = wb[:n]
        bias = wb[n:] if ctx.has_bias else None
        if g_logp is None and g_entropy is None:
            return (None,) * (6 + len(wb))
        g = _f32(g_logp) if g_logp is not None else _zeros_like_rows(X)
        want_db = bias is not None and any(b is not None and b.requires_grad for b in bias)
        # X and W are bf16, so their gradients are bf16: the library rounds its fp32 results
        # once, as autograd's own cast would, and writes half the bytes
        r = lp_backward_ex(X, W, bias, ctx.part, y, ctx.tau, lse, g, bias_grad=want_db,
                           entropy=entropy if g_entropy is not None else None, grad_entropy=_f32(g_entropy),
                           dx_dtype=torch.bfloat16, dw_dtype=torch.bfloat16)
        dX = r["dX"] if ctx.needs_input_grad[0] else None
        dW = [d if ctx.needs_input_grad[6 + k] else None for k, d in enumerate(r["dW"])]
        db = [None] * n
        if want_db:
            db = [d if ctx.needs_input_grad[6 + n + k] else None for k, d in enumerate(r["db"])]
        return (dX, None, None, None, None, None, *dW, *(db if ctx.has_bias else []))


def linear_logp(X: torch.Tensor, W: Sequence[torch.Tensor], bias: Optional[Sequence[torch.Tensor]], part,
                y: torch.Tensor, tau: float):
    """Fused linear-logp with autograd: returns (logp, entropy), both differentiable with
    respect to X, every W[k] and every bias[k]. The merged LSE is kept for the backward."""
    n = len(part.ranges)
    if len(W) != n:
        raise ValueError("W must have one entry per shard")
    wb = list(W) + (list(bias) if bias is not None else [])
    logp, entropy, _ = _LinearLogp.apply(X, part, y, float(tau), n, bias is not None, *wb)
    return logp, entropy


class _LinearLogpFromLogits(torch.autograd.Function):
    @staticmethod
    def forward(ctx, part, y, tau, *logits):
        out = lp_forward_from_logits(list(logits), part, y, tau, entropy=True)
        ctx.part, ctx.tau = part, tau
        ctx.save_for_backward(y, out["lse"], out["entropy"], *logits)
        ctx.mark_non_differentiable(out["lse"])
        ctx.set_materialize_grads(False)
        return out["logp"], out["entropy"], out["lse"]

    @staticmethod
    def backward(ctx, g_logp, g_entropy, _g_lse):
        y, lse, entropy, *logits = ctx.saved_tensors
        if g_logp is None and g_entropy is None:
            return (None,) * (3 + len(logits))
        g = _f32(g_logp) if g_logp is not None else _zeros_like_rows(y)
        dL = lp_backward_from_logits(logits, ctx.part, y, ctx.tau, lse, g,
                                     entropy=entropy if g_entropy is not None else None,
                                     grad_entropy=_f32(g_entropy), out_dtype=torch.bfloat16)
        return (None, None, None, *[d if ctx.needs_input_grad[3 + k] else None for k, d in enumerate(dL)])


def linear_logp_from_logits(logits: Sequence[torch.Tensor], part, y: torch.Tensor, tau: float):
    """Logits-reuse linear-logp with autograd: returns (logp, entropy), differentiable
    with respect to each shard's unscaled bf16 logits (gradients in bf16)."""
    if len(logits) != len(part.ranges):
        raise ValueError("logits must have one entry per shard")
    logp, entropy, _ = _LinearLogpFromLogits.apply(part, y, float(tau), *logits)
    return logp, entropy
