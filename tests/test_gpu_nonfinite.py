"""Non-finite logits.  -inf (a banned vocabulary entry) is a valid logit: it
adds exp(-inf) = 0 to the softmax sum and gets a zero gradient, and every
result must still match the oracle.  A NaN logit in a scored row makes that
row's lse, log-prob and gradient NaN and the loss NaN (the arithmetic
propagates it; nothing is reported as an error), while the other rows are
unaffected."""
import math

import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _banned_columns(w, ids, k, seed=0):
    """k vocabulary columns that no completion token uses (so no target is -inf)."""
    used = set(np.unique(ids[:, w.P:]).tolist())
    free = np.array([v for v in range(w.V) if v not in used])
    rng = np.random.default_rng(seed)
    return rng.choice(free, size=min(k, len(free)), replace=False)


@pytest.mark.parametrize("dtype,V", [("f32", 1024), ("bf16", 4099)])
@pytest.mark.parametrize("fused", [False, True], ids=["two_pass", "fused"])
def test_neg_inf_logits_match_oracle(dtype, V, fused):
    w = H.with_contrast(wl.variant(wl.TINY, name=f"neginf_{dtype}", dtype=dtype, V=V,
                                   old_sigma=0.1, ref_sigma=0.1, beta=0.04))
    ids = wl.make_ids(w)
    logits = wl.make_logits_cpu(w)
    cols = torch.from_numpy(_banned_columns(w, ids, V // 8))
    logits[:, :, cols] = float("-inf")
    logits[0, :, :] = float("-inf")  # completion 0: every non-target column banned ...
    for t in range(w.T - 1):         # ... except the token each row scores
        logits[0, t, int(ids[0, t + 1])] = 0.0
    out, _ = H.check_small(w, logits_cpu=logits, fused=fused)
    d = out["dlogits"].float().cpu()
    assert torch.all(d[:, :, cols] == 0)


@pytest.mark.parametrize("fused", [False, True], ids=["two_pass", "fused"])
def test_nan_logit_propagates_to_its_row(fused):
    n = H.g()
    w = wl.variant(wl.TINY, name="nan_logit", dtype="bf16", V=3000)
    ids = wl.make_ids(w)
    logits = wl.make_logits_cpu(w)
    i, t = 1, 0                       # completion 1, token 0: logits row P-1
    y = int(ids[i, w.P + t])
    logits[i, w.P - 1, (y + 17) % w.V] = float("nan")
    z, dt = wl.logits_as_numpy(logits)
    _, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    lp_o, lse_o = oracle.logp(z, dt, w.P, w.C, ids, len_o)
    R = wl.make_rewards(w)
    # old log-probs = the oracle's (NaN at the NaN row): the ratio, and so the
    # loss, then depend on the log-probs (without old log-probs r is exactly 1)
    old = lp_o.astype(np.float32)
    out = H.run_gpu(w, logits.cuda(), ids, R, old, None, beta=0.0, fused=fused)
    assert out["status"] == 0
    lp = out["logp"].cpu().numpy()
    lse = out["lse"].cpu().numpy()
    assert math.isnan(lp[i, t]) and math.isnan(lse[i, t])
    assert math.isnan(float(out["loss"].item()))
    ok = np.ones(lp.shape, bool)
    ok[i, t] = False
    ok &= np.arange(w.C)[None, :] < len_o[:, None]
    assert np.max(np.abs(lp[ok] - lp_o[ok])) <= H.LOGP_ATOL["bf16"]
    d = out["dlogits"].float().cpu().numpy()
    assert np.all(np.isnan(d[i, w.P - 1]))
    others = np.ones((w.N, w.T), bool)
    others[i, w.P - 1] = False
    assert np.all(np.isfinite(d[others]))
