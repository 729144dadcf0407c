"""grpo_loss_fwd_static: the forward pass for callers that cannot allocate
device memory (inside an allocator or memory pool that must not be
re-entered, in a plugin host that only lends its own buffers, or in a runtime
that forbids allocation after start-up).  It uses a scratch array built into
the library instead of a caller-provided workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test.  The GPU test calls the new entry point through
the C ABI twice in a row and requires both results to have the bits of
grpo_loss_fwd's (the same kernels on the same workspace layout), which is
itself checked against the float64 oracle with the parity tolerances of the
other tests; the CPU test checks that a batch larger than the built-in
scratch is refused before any CUDA call."""
import ctypes

import numpy as np
import pytest

import oracle
from vocab_wide_logprob_gb300 import workloads as wl

STATIC_MAX_N = 4096


def test_static_entry_rejects_oversized_batch():
    from vocab_wide_logprob_gb300 import build
    lib = ctypes.CDLL(build.build())
    fn = lib.grpo_loss_fwd_static
    P, I64, F, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    fn.argtypes = [P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P, P]
    fn.restype = INT
    a = ctypes.c_void_p(0x10000)
    rc = fn(a, 1, STATIC_MAX_N + 1, 4, 8, 64, a, a, a, None, None, 0.2, 0.0, 0.0, a, a, a, a,
            None)
    assert rc == 2  # GRPO_ERR_UNSUPPORTED: larger than the built-in scratch


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_twice():
    import torch
    import gpu_harness as H
    from vocab_wide_logprob_gb300 import _native as g

    assert torch.cuda.is_available()
    w = H.with_contrast(wl.variant(wl.QWEN_G8, name="static", B=2, G=4, P=8, C=40,
                                   reward_p=0.5, old_sigma=0.1, ref_sigma=0.1, beta=0.04,
                                   seed=404))
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    R = torch.from_numpy(wl.make_rewards(w)).cuda()
    _, lens = g.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = g.grpo_advantage(R, w.G)
    base = g.grpo_loss_fwd(logits, w.P, ids, lens, adv)
    n_old, n_ref = wl.make_noise(w)
    old = (base["logp"] + torch.from_numpy(n_old).float().cuda()).contiguous()
    ref = (base["logp"] + torch.from_numpy(n_ref).float().cuda()).contiguous()

    want = g.grpo_loss_fwd(logits, w.P, ids, lens, adv, old, ref, w.eps, w.beta)
    torch.cuda.synchronize()
    assert g.grpo_check_error(want["workspace"]) == 0
    # the existing entry point against the float64 oracle, with the parity
    # tolerances of the other tests
    z, dt = wl.logits_as_numpy(logits.cpu())
    _, len_o = oracle.mask(wl.make_ids(w), w.P, w.C, w.eos_id)
    lp_o, lse_o = oracle.logp(z, dt, w.P, w.C, wl.make_ids(w), len_o)
    A_o = oracle.advantage(wl.make_rewards(w), w.G)
    o64 = lambda t: t.cpu().numpy().astype(np.float64)
    loss_o, w_o, ell_o = oracle.loss(lp_o, o64(old), o64(ref), A_o, len_o, w.eps, w.beta)
    assert np.max(np.abs(o64(want["logp"]) - lp_o)) <= H.LOGP_ATOL["bf16"]
    assert np.max(np.abs(o64(want["lse"]) - lse_o)) <= H.LOGP_ATOL["bf16"]
    H.assert_loss(float(want["loss"].item()), loss_o, ell_o, float(w.N * w.C))
    # the static-scratch entry point runs the same kernels on the same
    # workspace layout: its outputs must have exactly the same bits, on two
    # calls in a row (the second finds the first call's scratch contents)
    for _ in range(2):
        got = g.grpo_loss_fwd_static(logits, w.P, ids, lens, adv, old, ref, w.eps, w.beta)
        torch.cuda.synchronize()
        for k in ("logp", "lse", "w", "loss"):
            assert torch.equal(got[k].view(torch.int32), want[k].view(torch.int32)), k
