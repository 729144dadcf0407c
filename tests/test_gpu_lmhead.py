"""grpo_lmhead_logprobs (LM-head projection on the tensor cores fused with the
log-sum-exp and gather) against the float64 oracle: the logits hidden x W^T
in float64 from the same bf16 inputs, then log_softmax and gather."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = H.LOGP_ATOL["bf16"]


def _bits16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(w, d, device_gen=False):
    g = H.g()
    dev = "cuda" if device_gen else "cpu"
    hidden = wl.make_hidden(w, d, dev).cuda()
    weight = wl.make_lm_head(w, d, dev).cuda()
    ids = wl.make_ids(w)
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    lp, lse, ws = g.grpo_lmhead_logprobs(hidden, weight, w.P, t_ids, lens)
    status = g.grpo_check_error(ws)
    return hidden, weight, ids, lens.cpu().numpy(), lp.cpu().numpy(), lse.cpu().numpy(), status


@pytest.mark.parametrize("V,d", [(1000, 128), (1000, 256), (4099, 384), (151936, 896)])
def test_lmhead_small(V, d):
    w = wl.variant(wl.QWEN_G8, name=f"lm_{V}_{d}", B=1, G=4, P=8, C=24, V=V, seed=60 + d,
                   eos_id=min(wl.QWEN25_EOS, V - 1))
    hidden, weight, ids, lens, lp, lse, status = _run(w, d)
    assert status == 0
    lp_o, lse_o = oracle.lmhead_logp(_bits16(hidden), _bits16(weight), w.P, w.C, ids, lens)
    assert np.max(np.abs(lp - lp_o)) <= TOL, np.max(np.abs(lp - lp_o))
    assert np.max(np.abs(lse - lse_o)) <= TOL
    m = np.arange(w.C)[None, :] >= lens[:, None]
    assert np.all(lp[m] == 0) and np.all(lse[m] == 0)


def test_lmhead_full_size_default_workload():
    """The benchmark workload's shapes with Qwen2.5-0.5B's hidden size 896:
    989 scored rows (8 blocks of 128, split over the vocabulary), every
    log-prob checked."""
    w = wl.QWEN_G8
    hidden, weight, ids, lens, lp, lse, status = _run(w, 896, device_gen=True)
    assert status == 0
    lp_o, lse_o = oracle.lmhead_logp(_bits16(hidden), _bits16(weight), w.P, w.C, ids, lens)
    assert np.max(np.abs(lp - lp_o)) <= TOL, np.max(np.abs(lp - lp_o))
    assert np.max(np.abs(lse - lse_o)) <= TOL


def test_lmhead_many_row_blocks_sampled():
    """18,879 scored rows (148 blocks: one vocabulary split each): sampled rows
    against the oracle, and determinism across two calls."""
    w = wl.BATCHED
    g = H.g()
    hidden = wl.make_hidden(w, 896, "cuda")
    weight = wl.make_lm_head(w, 896, "cuda")
    ids = wl.make_ids(w)
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    lp, lse, ws = g.grpo_lmhead_logprobs(hidden, weight, w.P, t_ids, lens)
    lp2, lse2, _ = g.grpo_lmhead_logprobs(hidden, weight, w.P, t_ids, lens, workspace=ws)
    assert g.grpo_check_error(ws) == 0
    assert torch.equal(lp.view(torch.int32), lp2.view(torch.int32))
    L = lens.cpu().numpy()
    rng = np.random.default_rng(3)
    Wn = _bits16(weight)
    for _ in range(48):
        i = int(rng.integers(0, w.N))
        t = int(rng.integers(0, L[i]))
        h = _bits16(hidden[i, w.P - 1 + t:w.P + t])
        a, b = oracle.lmhead_logp(h[None], Wn, 1, 1, np.array([[0, ids[i, w.P + t]]]),
                                  np.array([1], np.int32))
        assert abs(lp[i, t].item() - a[0, 0]) <= TOL, (i, t, lp[i, t].item(), a[0, 0])
        assert abs(lse[i, t].item() - b[0, 0]) <= TOL


def test_lmhead_bad_token_reported():
    w = wl.variant(wl.QWEN_G8, name="lm_bad", B=1, G=4, P=8, C=24, V=1000, eos_id=999, seed=5)
    g = H.g()
    hidden = wl.make_hidden(w, 128).cuda()
    weight = wl.make_lm_head(w, 128).cuda()
    ids = wl.make_ids(w)
    ids[0, w.P + 2] = 5000
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    lp, _, ws = g.grpo_lmhead_logprobs(hidden, weight, w.P, t_ids, lens)
    assert g.grpo_check_error(ws) == 6
    assert np.isnan(lp[0, 2].item())


@pytest.mark.parametrize("V,d,B,G,C", [(200, 128, 1, 2, 3), (256, 128, 1, 1, 1), (257, 256, 2, 2, 5)],
                         ids=["V_below_tile", "one_row", "V_tile_plus_one"])
def test_lmhead_edge_shapes(V, d, B, G, C):
    w = wl.variant(wl.QWEN_G8, name=f"lm_edge_{V}", B=B, G=G, P=3, C=C, V=V, eos_id=V - 1,
                   seed=70 + V)
    hidden, weight, ids, lens, lp, lse, status = _run(w, d)
    assert status == 0
    lp_o, lse_o = oracle.lmhead_logp(_bits16(hidden), _bits16(weight), w.P, w.C, ids, lens)
    assert np.max(np.abs(lp - lp_o)) <= TOL and np.max(np.abs(lse - lse_o)) <= TOL


def test_lmhead_empty_batch():
    g = H.g()
    hidden = torch.zeros((0, 6, 128), dtype=torch.bfloat16, device="cuda")
    weight = torch.zeros((300, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, 6), dtype=torch.int64, device="cuda")
    lens = torch.zeros((0,), dtype=torch.int32, device="cuda")
    lp, lse, ws = g.grpo_lmhead_logprobs(hidden, weight, 2, ids, lens)
    assert lp.numel() == 0 and g.grpo_check_error(ws) == 0
