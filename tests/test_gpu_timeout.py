"""The kernels' bounded waits end by themselves: a wait on a barrier that
nothing completes gives up after its one-second limit, records the timeout
in the workspace, and leaves the context usable (no fault, trap or hang)."""
import time

import pytest
import torch

import gpu_harness as H
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GRPO_ERR_TIMEOUT = 8


def test_bounded_wait_gives_up_and_reports():
    n = H.g()
    w = wl.TINY
    ws = torch.zeros((n.grpo_workspace_size(w.N, w.C, w.V),), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    n.grpo_selftest_timeout(ws)
    assert n.grpo_check_error(ws) == GRPO_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.9 <= elapsed < 30, elapsed

    # the context is still usable, and a loss forward on the same workspace
    # resets its error flags
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(torch.from_numpy(wl.make_rewards(w)).cuda(), w.G)
    n.grpo_loss_fwd(logits, w.P, ids, lens, adv, workspace=ws)
    assert n.grpo_check_error(ws) == 0
    H.check_small(w)
