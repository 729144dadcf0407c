"""The torch.autograd binding: loss.backward() gives the oracle's d loss /
d logits (and the bits of grpo_loss_bwd), scaled by the upstream gradient."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl
from vocab_wide_logprob_gb300.autograd import grpo_loss

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("scale", [1.0, 3.0])
def test_backward_matches_oracle(scale):
    w = H.with_contrast(wl.variant(wl.TINY, name="autograd", old_sigma=0.1, ref_sigma=0.1,
                                   beta=0.04))
    n = H.g()
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    logits_cpu = wl.make_logits_cpu(w)
    z, dt = wl.logits_as_numpy(logits_cpu)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage(R, w.G)
    lp_o, lse_o = oracle.logp(z, dt, w.P, w.C, ids, len_o)
    old, ref = H.host_inputs(w, lp_o, m_o)
    nrm = float(w.N * w.C)
    loss_o, w_o, ell_o = oracle.loss(lp_o, old.astype(np.float64), ref.astype(np.float64), A_o,
                                     len_o, w.eps, w.beta, nrm)
    d_o = oracle.dlogits(z, dt, w.P, w.C, ids, len_o, lse_o, w_o, scale)

    t_ids = H.dev(ids)
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(R), w.G)
    logits = logits_cpu.cuda().requires_grad_(True)
    loss = grpo_loss(logits, w.P, t_ids, lens, adv, H.dev(old), H.dev(ref), w.eps, w.beta)
    assert loss.shape == () and loss.requires_grad
    (loss * scale).backward()
    H.assert_loss(float(loss.item()), loss_o, ell_o, nrm)
    kink = H.kink_tokens(lp_o, old, w.eps)
    rows_ok = np.ones((w.N, w.T), bool)
    for i, t in zip(*np.nonzero(kink)):
        rows_ok[i, w.P - 1 + t] = False
    d = logits.grad.float().cpu().numpy()
    H.assert_dlogits(d[rows_ok], d_o[rows_ok], "autograd")

    # the same bits as the two C-ABI calls with the upstream gradient passed in
    out = n.grpo_loss_fwd(logits.detach(), w.P, t_ids, lens, adv, H.dev(old), H.dev(ref), w.eps,
                          w.beta)
    gt = torch.tensor([scale], dtype=torch.float32, device="cuda")
    dl = n.grpo_loss_bwd(logits.detach(), w.P, t_ids, lens, out["lse"], out["w"], gt)
    torch.cuda.synchronize()
    assert torch.equal(dl.view(torch.int32), logits.grad.view(torch.int32))


def test_bf16_logits_grad_dtype_and_shape():
    w = H.with_contrast(wl.variant(wl.TINY, name="autograd_bf16", dtype="bf16", V=4099))
    n = H.g()
    t_ids = H.dev(wl.make_ids(w))
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(wl.make_rewards(w)), w.G)
    logits = wl.make_logits_cpu(w).cuda().requires_grad_(True)
    grpo_loss(logits, w.P, t_ids, lens, adv).backward()
    assert logits.grad.dtype == torch.bfloat16 and logits.grad.shape == logits.shape
    out = n.grpo_loss_fwd(logits.detach(), w.P, t_ids, lens, adv)
    dl = n.grpo_loss_bwd(logits.detach(), w.P, t_ids, lens, out["lse"], out["w"])
    torch.cuda.synchronize()
    assert torch.equal(dl.view(torch.int16), logits.grad.view(torch.int16))
