"""torch.autograd bindings of the loss: the forward is grpo_loss_fwd, the
backward grpo_loss_bwd (d loss / d logits, "loss.backward()" of "Making Dr
GRPO go brrr", salahadawi.com), both through the C ABI; torch only holds
the tensors.  GRPOLMHeadLoss does the same from hidden states and the LM head
(grpo_lmhead_loss_fwd / grpo_lmhead_loss_bwd).

Only the logits (or the hidden states and the LM head) receive a gradient.  The advantages, old and reference
log-probs are constants of the update step (the advantage comes from the
rewards, the old and reference log-probs from no-grad passes), so their
gradients are None.
"""
from __future__ import annotations

import torch

from . import _native as g


class GRPOLoss(torch.autograd.Function):
    """loss = GRPOLoss.apply(logits, P, input_ids, lens, adv, old_logp,
    ref_logp, eps, beta, norm, agg): a 0-dim float32 tensor on the logits'
    device; ``loss.backward()`` writes d loss / d logits (same dtype and shape
    as the logits) scaled by the upstream gradient."""

    @staticmethod
    def forward(ctx, logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2,
                beta=0.0, norm=0.0, agg=None):
        out = g.grpo_loss_fwd(logits, P, input_ids, lens, adv, old_logp, ref_logp, eps, beta,
                              norm, agg=agg)
        ctx.save_for_backward(logits, input_ids, lens, out["lse"], out["w"])
        ctx.P = P
        return out["loss"].reshape(())

    @staticmethod
    def backward(ctx, grad_loss):
        logits, input_ids, lens, lse, w = ctx.saved_tensors
        gl = grad_loss.detach().reshape(1).to(torch.float32).contiguous()
        dlogits = g.grpo_loss_bwd(logits, ctx.P, input_ids, lens, lse, w, gl)
        return (dlogits,) + (None,) * 10


def grpo_loss(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2, beta=0.0,
              norm=0.0, agg=None):
    """Functional form of :class:`GRPOLoss` (differentiable in ``logits``)."""
    return GRPOLoss.apply(logits, P, input_ids, lens, adv, old_logp, ref_logp, eps, beta, norm,
                          agg)


class GRPOLMHeadLoss(torch.autograd.Function):
    """loss = GRPOLMHeadLoss.apply(hidden, weight, P, input_ids, lens, adv,
    old_logp, ref_logp, eps, beta, norm, agg, rows_per_pass): the loss from
    hidden states [N, P+C, d] and the LM head [V, d] (both bfloat16), the
    projection fused on the tensor cores (grpo_lmhead_loss_fwd); the logits
    are never written.  ``loss.backward()`` writes d loss / d hidden and
    d loss / d weight (grpo_lmhead_loss_bwd, computed in float32 and handed
    to autograd, which stores them in the parameters' dtype), scaled by the
    upstream gradient.

    ``rows_per_pass``: rows per pass of the backward's workspace.  None (the
    default) takes the number of scored rows, read on the host from ``lens``
    (one synchronisation per backward), so that one pass covers them; 0 sizes
    it for every possible row (no synchronisation, N·C·V·2 bytes of logits
    gradient buffer)."""

    @staticmethod
    def forward(ctx, hidden, weight, P, input_ids, lens, adv, old_logp=None, ref_logp=None,
                eps=0.2, beta=0.0, norm=0.0, agg=None, rows_per_pass=None):
        out = g.grpo_lmhead_loss_fwd(hidden, weight, P, input_ids, lens, adv, old_logp, ref_logp,
                                     eps, beta, norm, agg=agg)
        ctx.save_for_backward(hidden, weight, input_ids, lens, out["lse"], out["w"])
        ctx.P = P
        ctx.rows_per_pass = rows_per_pass
        return out["loss"].reshape(())

    @staticmethod
    def backward(ctx, grad_loss):
        hidden, weight, input_ids, lens, lse, w = ctx.saved_tensors
        gl = grad_loss.detach().reshape(1).to(torch.float32).contiguous()
        rpp = ctx.rows_per_pass
        if rpp is None:
            rpp = max(1, int(lens.sum().item()))
        dh, dw, _ = g.grpo_lmhead_loss_bwd(hidden, weight, ctx.P, input_ids, lens, lse, w, gl,
                                           rows_per_pass=rpp)
        return (dh, dw) + (None,) * 11


def grpo_lmhead_loss(hidden, weight, P, input_ids, lens, adv, old_logp=None, ref_logp=None,
                     eps=0.2, beta=0.0, norm=0.0, agg=None, rows_per_pass=None):
    """Functional form of :class:`GRPOLMHeadLoss` (differentiable in
    ``hidden`` and ``weight``)."""
    return GRPOLMHeadLoss.apply(hidden, weight, P, input_ids, lens, adv, old_logp, ref_logp, eps,
                                beta, norm, agg, rows_per_pass)
