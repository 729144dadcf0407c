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


@pytest.mark.parametrize("rows_per_pass", [None, 0], ids=["scored_rows", "every_row"])
def test_lmhead_backward_gives_the_c_abi_gradients(rows_per_pass):
    """GRPOLMHeadLoss: the loss of grpo_lmhead_loss_fwd, and loss.backward()
    stores grpo_lmhead_loss_bwd's dhidden and dweight (whose parity with the
    oracle the LM-head gradient tests establish) in the parameters' bf16,
    scaled by the upstream gradient."""
    from vocab_wide_logprob_gb300.autograd import grpo_lmhead_loss
    w = H.with_contrast(wl.variant(wl.QWEN_G8, name="autograd_lm", B=2, G=4, P=8, C=24, V=1000,
                                   eos_id=999, seed=81))
    d = 128
    n = H.g()
    ids = H.dev(wl.make_ids(w))
    _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(wl.make_rewards(w)), w.G)
    gen = torch.Generator().manual_seed(5)
    hidden = torch.randn((w.N, w.T, d), generator=gen).to(torch.bfloat16).cuda()
    weight = (torch.randn((w.V, d), generator=gen) * 0.05).to(torch.bfloat16).cuda()
    hidden.requires_grad_(True)
    weight.requires_grad_(True)
    loss = grpo_lmhead_loss(hidden, weight, w.P, ids, lens, adv, rows_per_pass=rows_per_pass)
    assert loss.shape == () and loss.requires_grad
    (loss * 2.0).backward()

    f = n.grpo_lmhead_loss_fwd(hidden.detach(), weight.detach(), w.P, ids, lens, adv)
    gt = torch.tensor([2.0], dtype=torch.float32, device="cuda")
    rpp = int(lens.sum().item()) if rows_per_pass is None else rows_per_pass
    dh, dw, _ = n.grpo_lmhead_loss_bwd(hidden.detach(), weight.detach(), w.P, ids, lens,
                                       f["lse"], f["w"], gt, rows_per_pass=rpp)
    torch.cuda.synchronize()
    assert torch.equal(loss.detach().reshape(1).view(torch.int32), f["loss"].view(torch.int32))
    assert hidden.grad.dtype == torch.bfloat16 and weight.grad.dtype == torch.bfloat16
    assert torch.equal(hidden.grad.view(torch.int16), dh.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(weight.grad.view(torch.int16), dw.to(torch.bfloat16).view(torch.int16))
    assert float(dw.abs().sum()) > 0  # the group has reward contrast: a live gradient
