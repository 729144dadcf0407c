"""GB300 (sm_103a) Dr. GRPO loss over policy logits, forward and backward.

The compute lives in ``libgrpo.so`` (hand-written CUDA kernels behind the C
ABI in ``include/grpo.h``); :mod:`vocab_wide_logprob_gb300._native` is its
thin ctypes binding and :mod:`vocab_wide_logprob_gb300.workloads` draws the
seeded synthetic inputs.  The binding is imported lazily so that the input
generators stay usable on machines without the built library.
"""

_NAMES = ("grpo_mask", "grpo_advantage", "grpo_advantage_ex", "grpo_workspace_size",
          "grpo_loss_fwd", "grpo_loss_fwd_ex", "grpo_logprobs", "grpo_loss_bwd",
          "grpo_loss_bwd_ex", "grpo_loss_fwd_bwd", "grpo_loss_fwd_bwd_ex", "grpo_loss_fwd_bwd_host",
          "grpo_loss_fwd_static",
          "grpo_lmhead_logprobs", "grpo_lmhead_loss_fwd", "grpo_lmhead_loss_bwd",
          "grpo_check_error", "grpo_selftest_timeout", "grpo_set_early_start", "grpo_copy", "GrpoError")


def __getattr__(name):
    if name in _NAMES:
        from . import _native
        return getattr(_native, name)
    if name in ("GRPOLoss", "grpo_loss"):
        from . import autograd
        return getattr(autograd, name)
    raise AttributeError(name)
