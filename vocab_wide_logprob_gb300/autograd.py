"""torch.autograd binding of the loss: the forward is grpo_loss_fwd, the
backward grpo_loss_bwd (d loss / d logits, "loss.backward()" of "Making Dr
GRPO go brrr", salahadawi.com), both through the C ABI; torch only holds
the tensors.

Only the logits receive a gradient.  The advantages, old and reference
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
