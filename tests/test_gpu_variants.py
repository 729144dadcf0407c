"""The original-GRPO options, the log-prob-only pass and the zero-weight skip
against the float64 oracle (and against the default path where they must
agree bit for bit)."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("G", [1, 3, 4, 8, 16, 32, 40])
def test_advantage_std_and_contrast_count(G):
    g = H.g()
    rng = np.random.default_rng(G)
    B = 37
    for R in (rng.integers(0, 2, size=B * G).astype(np.float32),
              rng.normal(0, 2, size=B * G).astype(np.float32)):
        R[:G] = 1.0  # one uniform group
        A_o = oracle.advantage_std(R, G, 1e-4)
        adv, cnt = g.grpo_advantage_ex(torch.from_numpy(R).cuda(), G, 1, 1e-4, count_contrast=True)
        a = adv.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(a - A_o) <= 2e-6 * np.maximum(1.0, np.abs(A_o))), np.max(np.abs(a - A_o))
        assert int(cnt.item()) == oracle.contrast_count(R, G)
        # mode 0 is grpo_advantage, bit for bit
        a0, c0 = g.grpo_advantage_ex(torch.from_numpy(R).cuda(), G, 0, 0.0, count_contrast=True)
        assert torch.equal(a0, g.grpo_advantage(torch.from_numpy(R).cuda(), G))
        assert int(c0.item()) == int(cnt.item())


def _variant_check(w, agg, adv_mode, fused, grad=None):
    g = H.g()
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    logits_cpu = wl.make_logits_cpu(w)
    z, dt = wl.logits_as_numpy(logits_cpu)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage_std(R, w.G, 1e-4) if adv_mode else oracle.advantage(R, w.G)
    lp_o, lse_o = oracle.logp(z, dt, w.P, w.C, ids, len_o)
    old, ref = H.host_inputs(w, lp_o, m_o)
    o64 = lambda x: None if x is None else x.astype(np.float64)
    if agg:
        loss_o, w_o, ell_o = oracle.loss_seq_mean(lp_o, o64(old), o64(ref), A_o, len_o, w.eps,
                                                  w.beta)
        nrm = float(w.N)
    else:
        loss_o, w_o, ell_o = oracle.loss(lp_o, o64(old), o64(ref), A_o, len_o, w.eps, w.beta)
        nrm = float(w.N * w.C)
    gval = 1.0 if grad is None else grad
    d_o = oracle.dlogits(z, dt, w.P, w.C, ids, len_o, lse_o, w_o, gval)

    logits = logits_cpu.cuda()
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv, _ = g.grpo_advantage_ex(torch.from_numpy(R).cuda(), w.G, adv_mode, 1e-4)
    gt = None if grad is None else torch.tensor([grad], device="cuda")
    if fused:
        out = g.grpo_loss_fwd_bwd_ex(logits, w.P, t_ids, lens, adv, H.dev(old), H.dev(ref), w.eps,
                                     w.beta, 0.0, agg, gt)
        dl = out["dlogits"]
    else:
        out = g.grpo_loss_fwd_ex(logits, w.P, t_ids, lens, adv, H.dev(old), H.dev(ref), w.eps,
                                 w.beta, 0.0, agg)
        dl = g.grpo_loss_bwd(logits, w.P, t_ids, lens, out["lse"], out["w"], gt)
    assert g.grpo_check_error(out["workspace"]) == 0
    lp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lp - lp_o)) <= H.LOGP_ATOL[dt]
    H.assert_loss(float(out["loss"].item()), loss_o, ell_o, nrm)
    kink = H.kink_tokens(lp_o, old, w.eps)
    rows_ok = np.ones((w.N, w.T), bool)
    for i, t in zip(*np.nonzero(kink)):
        rows_ok[i, w.P - 1 + t] = False
    H.assert_dlogits(dl.float().cpu().numpy()[rows_ok], d_o[rows_ok], w.name)
    return out, dl


CASES = [
    wl.variant(wl.TINY, name="tiny_v", old_sigma=0.1, ref_sigma=0.1, beta=0.04, reward_p=0.5),
    wl.variant(wl.QWEN_G8, name="bf16_v", B=2, G=4, P=8, C=24, reward_p=0.5, old_sigma=0.1,
               ref_sigma=0.1, beta=0.04, trunc=0.25, seed=78),
]


@pytest.mark.parametrize("fused", [False, True], ids=["two_pass", "fused"])
@pytest.mark.parametrize("agg,adv_mode", [(1, 0), (0, 1), (1, 1)],
                         ids=["seq_mean", "std_adv", "seq_mean_std_adv"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_original_grpo_options(w, agg, adv_mode, fused):
    _variant_check(H.with_contrast(w), agg, adv_mode, fused, grad=3.0)


def test_seq_mean_fused_same_bits():
    w = H.with_contrast(CASES[1])
    a, da = _variant_check(w, 1, 0, False)
    b, db = _variant_check(w, 1, 0, True)
    for k in ("logp", "lse", "w"):
        assert torch.equal(_bits(a[k]), _bits(b[k])), k
    assert torch.equal(_bits(da), _bits(db))


@pytest.mark.parametrize("w", [wl.TINY, CASES[1],
                               wl.variant(wl.TINY, name="lp_N1100", B=275, G=4, P=2, C=3, V=64),
                               wl.variant(wl.TINY, name="lp_N4100", B=1025, G=4, P=2, C=3, V=64)],
                         ids=lambda w: w.name)
def test_logprobs_only(w):
    """The log-probs-only call gives the loss forward's logp and lse bits and
    0 past each length; 1,100 completions build the length prefix table in
    each CTA, 4,100 read the one prep writes."""
    g = H.g()
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    _, lens = g.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = torch.zeros((w.N,), device="cuda")
    full = g.grpo_loss_fwd(logits, w.P, ids, lens, adv)
    lp, lse, ws = g.grpo_logprobs(logits, w.P, ids, lens)
    assert g.grpo_check_error(ws) == 0
    assert torch.equal(_bits(lp), _bits(full["logp"])) and torch.equal(_bits(lse), _bits(full["lse"]))
    _, len_o = oracle.mask(wl.make_ids(w), w.P, w.C, w.eos_id)
    past = np.arange(w.C)[None, :] >= len_o[:, None]
    assert past.any() and not past.all()
    assert np.all(_bits(lp).cpu().numpy()[past] == 0) and np.all(_bits(lse).cpu().numpy()[past] == 0)


SKIP_CASES = [
    # no reward contrast, beta = 0: every gradient weight is exactly 0
    wl.variant(wl.QWEN_G8, name="skip_nc", B=1, G=4, P=8, C=24, seed=5,
               forced={"rewards": [0.0] * 4}, old_sigma=0.1),
    # two groups, one with contrast: zero-weight rows beside live ones
    wl.variant(wl.QWEN_G8, name="skip_c", B=2, G=4, P=8, C=24, reward_p=0.5, old_sigma=0.1,
               seed=6, forced={"rewards": [1.0, 0.0, 0.0, 1.0, 1.0, 1.0, 1.0, 1.0]}),
    # beta > 0: the KL term keeps every weight nonzero, nothing is skipped
    wl.variant(wl.QWEN_G8, name="skip_kl", B=2, G=4, P=8, C=24, reward_p=0.5, old_sigma=0.1,
               ref_sigma=0.1, beta=0.04, seed=7, forced={"rewards": [1.0] * 8}),
    # float32 logits, ragged vocabulary
    wl.variant(wl.TINY, name="skip_f32", V=1003, old_sigma=0.1, reward_p=0.5, seed=8),
]


@pytest.mark.parametrize("w", SKIP_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("grad", [None, 7.0], ids=["g1", "g7"])
def test_skip_zero_weight_against_oracle(w, grad):
    """The backward with GRPO_BWD_SKIP_ZERO_WEIGHT against the float64 oracle,
    element by element over the whole batch (the rows it skips are compared
    like every other row)."""
    out, o = H.check_small(w, grad=grad, bwd_flags=1)
    nonzero = int((out["w"] != 0).sum().item())
    assert (nonzero == 0) == (w.name == "skip_nc"), (w.name, nonzero)
    if w.name == "skip_c":
        assert 0 < nonzero < int(out["lens"].sum().item())


def test_skip_zero_weight():
    """No reward contrast and beta = 0: every w is 0, so with the skip flag the
    gradient is written as +0 without reading any logits; with contrast the
    skip changes nothing but the sign of zero on zero-weight rows."""
    g = H.g()
    for w, contrast in ((wl.variant(wl.QWEN_G8, name="nc", B=1, G=4, P=8, C=24, seed=5,
                                    forced={"rewards": [0.0] * 4}, old_sigma=0.1), False),
                        (H.with_contrast(wl.variant(wl.QWEN_G8, name="c", B=2, G=4, P=8, C=24,
                                                    reward_p=0.5, old_sigma=0.1, seed=6)),
                         True)):
        logits = wl.make_logits_cpu(w).cuda()
        ids = torch.from_numpy(wl.make_ids(w)).cuda()
        _, lens = g.grpo_mask(ids, w.P, w.C, w.eos_id)
        adv = g.grpo_advantage(torch.from_numpy(wl.make_rewards(w)).cuda(), w.G)
        out = g.grpo_loss_fwd(logits, w.P, ids, lens, adv)
        a = g.grpo_loss_bwd(logits, w.P, ids, lens, out["lse"], out["w"])
        b = g.grpo_loss_bwd_ex(logits, w.P, ids, lens, out["lse"], out["w"], flags=1)
        torch.cuda.synchronize()
        assert torch.equal(a.float(), b.float())  # -0 == +0
        if not contrast:
            assert torch.all(_bits(b) == 0)  # +0 everywhere: nothing was read
