"""Rows split over a thread block cluster.  The log-sum-exp kernels give a
whole row to one CTA when the batch has enough rows to occupy the GPU, and
split each row over K = 2, 4 or 8 CTAs of a cluster (partials merged through
distributed shared memory) when N*C * K first reaches 4 x 152 SMs.  These
Qwen-vocabulary batches are sized to take K = 8, 4, 2 and 1 on a 152-SM
GB300; each is checked against the oracle on both paths, and the fused path
against the two calls bit for bit."""
import pytest
import torch

import gpu_harness as H
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


SIZES = [dict(B=1, G=2, C=40), dict(B=1, G=4, C=75), dict(B=1, G=4, C=125),
         dict(B=1, G=4, C=160)]
IDS = ["rows80_K8", "rows300_K4", "rows500_K2", "rows640_K1"]


def _w(kw):
    return H.with_contrast(wl.variant(wl.QWEN_G8, name=f"split_{kw['G'] * kw['C']}", P=4,
                                      reward_p=0.5, old_sigma=0.1, ref_sigma=0.1, beta=0.04,
                                      seed=300 + kw["C"], **kw))


@pytest.mark.parametrize("kw", SIZES, ids=IDS)
def test_split_matches_oracle(kw):
    w = _w(kw)
    logits_cpu = wl.make_logits_cpu(w)
    H.check_small(w, logits_cpu=logits_cpu)
    H.check_small(w, logits_cpu=logits_cpu, fused=True)


@pytest.mark.parametrize("kw", SIZES, ids=IDS)
def test_split_fused_same_bits(kw):
    w = _w(kw)
    logits = wl.make_logits_cpu(w).cuda()
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    a = H.run_gpu(w, logits, ids, R, None, None, grad=2.0, beta=0.0)
    b = H.run_gpu(w, logits, ids, R, None, None, grad=2.0, beta=0.0, fused=True)
    for k in ("logp", "lse", "w", "dlogits"):
        assert torch.equal(_bits(a[k]), _bits(b[k])), k
