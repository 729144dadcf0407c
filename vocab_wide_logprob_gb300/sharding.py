"""Data-parallel sharding of the Dr. GRPO loss path by prompt group.

Every quantity of the path is local to a prompt group (its G completions)
except the scalar loss, which is a token sum divided by a constant.  A rank
that holds whole groups and divides by the GLOBAL constant (pass it as the
``norm`` argument of ``grpo_loss_fwd``) produces a partial loss; the partials
of all ranks add up to the loss of the whole batch, and each rank's dlogits
are exactly the rows of the whole batch's dlogits for its completions.  The
only exchange is therefore one float (the loss, for reporting).
"""
from __future__ import annotations


def group_range(B: int, world: int, rank: int) -> range:
    """Prompt groups of `rank`: contiguous, sizes differ by at most one."""
    if not (0 <= rank < world):
        raise ValueError("rank outside [0, world)")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def completion_slice(B: int, G: int, world: int, rank: int) -> slice:
    """Completions (rows of logits / ids / rewards) held by `rank`."""
    r = group_range(B, world, rank)
    return slice(r.start * G, r.stop * G)


def global_norm(B: int, G: int, C: int) -> float:
    """The constant every rank divides its token sum by: N*C of the whole batch."""
    return float(B * G * C)
