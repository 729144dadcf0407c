"""Stream order of the backward.  Right after the loss forward on one stream,
grpo_loss_bwd writes the rows that score nothing before it waits on the
forward's last kernels (those rows depend only on the lengths), and the
scored rows after; after any other library call it waits first and walks the
rows in memory order.  Both orders must write every element with the same
bits, and the oracle must agree with the first (the parity tests run
forward -> backward back to back, so they take it too)."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def _both_orders(w, logits, flags=None, grad=None):
    n = H.g()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    R = torch.from_numpy(wl.make_rewards(w)).cuda()
    _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(R, w.G)
    gt = None if grad is None else torch.tensor([grad], dtype=torch.float32, device="cuda")
    # NaN-filled before the forward, so that no other kernel sits between the
    # forward and the first backward
    d_first = torch.full_like(logits, float("nan"))
    d_wait = torch.full_like(logits, float("nan"))
    out = n.grpo_loss_fwd(logits, w.P, ids, lens, adv, None, None, w.eps, 0.0)
    n.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"], gt, d_first, flags=flags)
    n.grpo_advantage(R, w.G, adv)  # a library call in between: the next backward waits first
    n.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"], gt, d_wait, flags=flags)
    assert n.grpo_check_error(out["workspace"]) == 0
    torch.cuda.synchronize()
    return d_first, d_wait, lens.cpu().numpy()


def _check(w, logits, **kw):
    d_first, d_wait, lens = _both_orders(w, logits, **kw)
    assert not torch.isnan(d_first).any() and not torch.isnan(d_wait).any()
    assert torch.equal(_bits(d_first), _bits(d_wait))
    # rows that score nothing are exactly +0 (bit pattern 0)
    zero = np.ones((w.N, w.T), bool)
    for i in range(w.N):
        zero[i, w.P - 1:w.P - 1 + int(lens[i])] = False
    zb = _bits(d_first)[torch.from_numpy(zero).cuda()]
    assert not bool((zb != 0).any())


@pytest.mark.parametrize("kw", [
    dict(),
    dict(C=1),
    dict(P=1),
    dict(B=1, G=32),
    dict(forced={"lengths": {i: 1 for i in range(8)}}),
    dict(forced={"lengths": {i: 0 for i in range(8)}}),
    dict(B=1, G=2, C=200, V=4099, dtype="bf16"),
], ids=["tiny", "C1", "P1", "G32", "eos_all", "eos_none", "C200_V4099_bf16"])
def test_orders_same_bits(kw):
    w = wl.variant(wl.TINY, name="order", **kw)
    _check(w, wl.make_logits_cpu(w).cuda())


def test_more_completions_than_the_prefix_table():
    """1,100 completions: above the 1,024 the reordered walk covers, so the
    backward waits first and walks memory order either way; the oracle agrees."""
    w = wl.variant(wl.TINY, name="order_n1100", B=275, G=4, P=2, C=3, V=64)
    _check(w, wl.make_logits_cpu(w).cuda())
    H.check_small(w)


def test_offsets_table_in_memory():
    """4,100 completions: the forward's log-sum-exp kernel reads the prefix
    table prep writes instead of building it in shared memory (it then waits
    on prep first); forward and backward still match the oracle and both
    backward orders agree."""
    w = wl.variant(wl.TINY, name="order_n4100", B=1025, G=4, P=2, C=3, V=64)
    _check(w, wl.make_logits_cpu(w).cuda())
    H.check_small(w)


def test_skip_zero_weight_orders_same_bits():
    w = wl.variant(wl.TINY, name="order_skip", B=4, G=4, C=40, V=2000, dtype="bf16")
    _check(w, wl.make_logits_cpu(w).cuda(), flags=1, grad=0.5)


def test_full_size_orders_same_bits():
    """The benchmark workload: the rows that score nothing (about two thirds
    of the 0.93 GB buffer) are written while the forward's kernels run."""
    w = wl.QWEN_G8
    logits = torch.empty((w.N, w.T, w.V), dtype=torch.bfloat16, device="cuda")
    wl.fill_logits_cuda(w, logits)
    _check(w, logits)


def test_no_scored_rows():
    """Every length 0: no CTA has a scored row, so only CTA 0 waits on the
    forward (before it exits); every element is written +0 either way."""
    n = H.g()
    w = wl.variant(wl.TINY, name="order_len0", dtype="bf16", V=3000)
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    lens = torch.zeros((w.N,), dtype=torch.int32, device="cuda")
    adv = n.grpo_advantage(torch.from_numpy(wl.make_rewards(w)).cuda(), w.G)
    d = torch.full_like(logits, float("nan"))
    out = n.grpo_loss_fwd(logits, w.P, ids, lens, adv)
    n.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"], None, d)
    assert n.grpo_check_error(out["workspace"]) == 0
    torch.cuda.synchronize()
    assert not bool((_bits(d) != 0).any())
    assert float(out["loss"].item()) == 0.0


@pytest.mark.parametrize("B", [256, 257], ids=["N1024_reordered", "N1028_memory_order"])
def test_prefix_table_boundary(B):
    """1,024 completions (the largest batch the reordered walk covers) and
    1,028 (memory order): same bits both ways, every element written."""
    w = wl.variant(wl.TINY, name=f"order_B{B}", B=B, G=4, P=2, C=3, V=64)
    _check(w, wl.make_logits_cpu(w).cuda())


def test_overlapping_buffers_wait_first():
    """dlogits carved from the same allocation as the forward's workspace (its
    first prompt rows, rows that score nothing, cover the workspace): in
    stream order the backward overwrites the workspace only after the forward
    is done with it.  The library sees the overlap and waits first, so the
    loss and dlogits equal those of separate buffers bit for bit."""
    n = H.g()
    w = H.with_contrast(wl.variant(wl.TINY, name="order_overlap", dtype="bf16", V=3000))
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    R = torch.from_numpy(wl.make_rewards(w)).cuda()
    _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(R, w.G)
    ref = n.grpo_loss_fwd(logits, w.P, ids, lens, adv, None, None, w.eps, 0.0)
    d_ref = n.grpo_loss_bwd(logits, w.P, ids, lens, ref["lse"], ref["w"], None)
    torch.cuda.synchronize()

    need = n.grpo_workspace_size(w.N, w.C, w.V)
    dl_bytes = logits.numel() * logits.element_size()
    # the workspace lies within sequence 0's prompt rows, which score nothing
    assert need <= (w.P - 1) * w.V * logits.element_size()
    buf = torch.full((dl_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    dl = buf.view(torch.bfloat16).view(logits.shape)
    ws = buf[:need]
    out = n.grpo_loss_fwd(logits, w.P, ids, lens, adv, None, None, w.eps, 0.0, workspace=ws)
    n.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"], None, dl)
    torch.cuda.synchronize()
    assert torch.equal(_bits(ref["loss"]), _bits(out["loss"]))
    for k in ("logp", "lse", "w"):
        assert torch.equal(_bits(ref[k]), _bits(out[k])), k
    assert torch.equal(_bits(d_ref), _bits(dl))


def test_early_starts_can_be_turned_off():
    """grpo_set_early_start(False): the backward and the advantage wait first
    like every launch; the results keep their bits."""
    n = H.g()
    w = H.with_contrast(wl.variant(wl.TINY, name="order_off", dtype="bf16", V=3000))
    logits = wl.make_logits_cpu(w).cuda()

    def run():
        ids = torch.from_numpy(wl.make_ids(w)).cuda()
        _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
        adv = n.grpo_advantage(torch.from_numpy(wl.make_rewards(w)).cuda(), w.G)
        out = n.grpo_loss_fwd(logits, w.P, ids, lens, adv)
        dl = n.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"])
        torch.cuda.synchronize()
        return adv, out, dl

    adv1, out1, dl1 = run()
    n.grpo_set_early_start(False)
    try:
        adv2, out2, dl2 = run()
    finally:
        n.grpo_set_early_start(True)
    assert torch.equal(adv1, adv2)
    for k in ("logp", "lse", "w", "loss"):
        assert torch.equal(_bits(out1[k]), _bits(out2[k])), k
    assert torch.equal(_bits(dl1), _bits(dl2))
