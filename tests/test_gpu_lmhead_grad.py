"""The loss through the LM head, forward (grpo_lmhead_loss_fwd) and backward
(grpo_lmhead_loss_bwd: gradients with respect to the hidden states and W on
the tensor cores) against the float64 oracle on the same bf16 inputs.

Tolerances, fixed from the arithmetic before looking at results:
* loss, w: as for the logits path (loss 1e-5 relative to max(|loss|, L1);
  w 1e-4 of the size of its terms);
* dhidden, dweight: the GPU rounds each logits-gradient entry dz to bf16
  (relative error <= 2^-9) before the float32 contractions, so each output
  element may move by at most 2^-9 times the sum of |dz| |operand| over its
  terms (the oracle's magnitude); the check allows 2^-7 of that magnitude
  (the rest covers float32 accumulation over up to V terms), requires exact
  zeros where the magnitude is 0, and bounds the relative Frobenius error of
  the whole sampled block by 1e-2.
Inputs whose oracle ratio lies near a clip boundary would let the two sides
take different branches of min() (and a dweight row sums over every token);
the old log-probs of such tokens are moved 2e-3 away on the host, for both
sides, before anything runs."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GRAD_MAG = 2.0 ** -7
GRAD_FRO = 1e-2


def _bits16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_grad(gpu, ref, mag, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = err > GRAD_MAG * mag
    assert not np.any(bad), (what, int(bad.sum()), np.argwhere(bad)[:5].tolist(),
                             float(np.max(err / np.maximum(mag, 1e-300))))
    nref = np.linalg.norm(ref)
    if nref > 0:
        assert np.linalg.norm(gpu - ref) <= GRAD_FRO * nref, (what, np.linalg.norm(gpu - ref) / nref)


def _setup(w, d, device_gen=False):
    n = H.g()
    gen = "cuda" if device_gen else "cpu"
    hidden = wl.make_hidden(w, d, gen).cuda()
    weight = wl.make_lm_head(w, d, gen).cuda()
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    Hn, Wn = _bits16(hidden), _bits16(weight)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage(R, w.G)
    lp_o, lse_o = oracle.lmhead_logp(Hn, Wn, w.P, w.C, ids, len_o)
    old, ref = H.host_inputs(w, lp_o, m_o)
    if old is not None:  # keep every ratio 1e-3 (log space) away from the clip boundaries
        kinks = np.array([-np.log1p(w.eps), -np.log1p(-w.eps)])
        with np.errstate(invalid="ignore"):
            dist = np.min(np.abs((old.astype(np.float64) - lp_o)[..., None] - kinks), axis=-1)
            old[dist < 1e-3] += np.float32(2e-3)
    assert not H.kink_tokens(lp_o, old, w.eps).any()
    nrm = float(w.N * w.C)
    loss_o, w_o, ell_o = oracle.loss(lp_o, None if old is None else old.astype(np.float64),
                                     None if ref is None else ref.astype(np.float64), A_o, len_o,
                                     w.eps, w.beta, nrm)
    t_ids = H.dev(ids)
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(R), w.G)
    out = n.grpo_lmhead_loss_fwd(hidden, weight, w.P, t_ids, lens, adv, H.dev(old), H.dev(ref),
                                 w.eps, w.beta)
    assert n.grpo_check_error(out["workspace"]) == 0
    host = dict(ids=ids, R=R, Hn=Hn, Wn=Wn, m=m_o, len=len_o, A=A_o, lp=lp_o, lse=lse_o, old=old,
                ref=ref, norm=nrm, loss=loss_o, w=w_o, ell=ell_o)
    return hidden, weight, t_ids, lens, out, host


def _check_fwd(w, out, h):
    lp = out["logp"].cpu().numpy().astype(np.float64)
    lse = out["lse"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lp - h["lp"])) <= H.LOGP_ATOL["bf16"]
    assert np.max(np.abs(lse - h["lse"])) <= H.LOGP_ATOL["bf16"]
    H.assert_loss(float(out["loss"].item()), h["loss"], h["ell"], h["norm"])
    wt = out["w"].cpu().numpy().astype(np.float64)
    scale = H.w_scale(h["lp"], h["old"], h["ref"], h["A"], w.beta, h["norm"])
    ok = h["m"] == 1
    assert np.all(np.abs(wt - h["w"])[ok] <= 1e-4 * scale[ok] + 1e-12)
    assert np.all(wt[~ok] == 0)


SMALL = [
    ("V1000_d128", wl.variant(wl.QWEN_G8, name="lmg_1000_128", B=2, G=4, P=8, C=24, V=1000,
                              eos_id=999, seed=81), 128, 1.0),
    ("V4099_d384_kl", wl.variant(wl.QWEN_G16_KL, name="lmg_4099_384", B=1, G=4, P=5, C=40,
                                 V=4099, eos_id=4000, seed=82), 384, 2.5),
    ("V300_d128_short", wl.variant(wl.QWEN_G8, name="lmg_300_128", B=1, G=2, P=3, C=6, V=300,
                                   eos_id=299, seed=83), 128, None),
    # several 512-column d tiles, the last one narrow, and more items than one
    # round of CTA pairs (dweight: 24 vocabulary blocks x 4 tiles; dhidden: 2
    # row blocks x 4 tiles x its vocabulary splits): four tiles rotate over
    # the rounds, three keep their order (a 152-SM grid's 76 pairs are not a
    # multiple of 3)
    ("V6001_d1664_four_tiles", wl.variant(wl.QWEN_G8, name="lmg_6001_1664", B=1, G=4, P=5,
                                          C=120, V=6001, eos_id=6000, seed=86), 1664, None),
    ("V6001_d1152_three_tiles", wl.variant(wl.QWEN_G8, name="lmg_6001_1152", B=1, G=4, P=5,
                                           C=120, V=6001, eos_id=6000, seed=87), 1152, 0.5),
    # a vocabulary smaller than one 256-column tile: the only tile runs past V
    ("V100_d128_subtile", wl.variant(wl.QWEN_G8, name="lmg_100_128", B=1, G=4, P=4, C=20,
                                     V=100, eos_id=99, seed=89), 128, 1.5),
    # Qwen2.5-7B's hidden size: seven 512-column d tiles, 56 k-steps per
    # projection tile
    ("V2000_d3584", wl.variant(wl.QWEN_G8, name="lmg_2000_3584", B=1, G=4, P=5, C=60, V=2000,
                               eos_id=1999, seed=88), 3584, None),
]


@pytest.mark.parametrize("name,w,d,g", SMALL, ids=[s[0] for s in SMALL])
def test_lmhead_grads_small(name, w, d, g):
    """Every element of the loss, w, dhidden and dweight against the oracle."""
    n = H.g()
    w = H.with_contrast(w)
    hidden, weight, t_ids, lens, out, h = _setup(w, d)
    _check_fwd(w, out, h)
    gt = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    dh, dw, ws = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                                        gt)
    assert n.grpo_check_error(ws) == 0
    gr = oracle.lmhead_grads(h["Hn"], h["Wn"], w.P, w.C, h["ids"], h["len"], h["lse"], h["w"],
                             1.0 if g is None else g, magnitudes=True)
    assert_grad(dh.cpu().numpy(), gr["dhidden"], gr["dhidden_mag"], "dhidden")
    assert_grad(dw.cpu().numpy(), gr["dweight"], gr["dweight_mag"], "dweight")


def test_lmhead_grads_deterministic_and_scaled():
    """Two calls give the same bits; an upstream gradient of 2 doubles every
    output exactly (bf16 rounding commutes with a power-of-two scale)."""
    n = H.g()
    w = H.with_contrast(SMALL[1][1])
    hidden, weight, t_ids, lens, out, h = _setup(w, 384)
    one = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    two = torch.tensor([2.0], dtype=torch.float32, device="cuda")
    a = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"], one)
    b = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"], one)
    c = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"], two)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    assert torch.equal(c[0], 2 * a[0]) and torch.equal(c[1], 2 * a[1])


def test_lmhead_grads_no_scored_rows():
    """C = 0: nothing is scored, both gradients are zero."""
    n = H.g()
    hidden = torch.ones((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    weight = torch.ones((300, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((2, 4), dtype=torch.int64, device="cuda")
    lens = torch.zeros((2,), dtype=torch.int32, device="cuda")
    z = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    dh, dw, ws = n.grpo_lmhead_loss_bwd(hidden, weight, 4, ids, lens, z, z)
    torch.cuda.synchronize()
    assert not dh.any() and not dw.any()


def test_lmhead_grads_full_size_default_workload():
    """The benchmark workload's shapes with Qwen2.5-0.5B's hidden size 896
    (about 1,000 scored rows, V = 151,936; the first seed with reward
    contrast): the forward against the oracle on every token; sampled rows of
    dhidden and sampled rows of dweight (the targets of some scored tokens
    among them) element by element; every row of dhidden that scores nothing
    exactly zero."""
    n = H.g()
    w = H.with_contrast(wl.QWEN_G8)
    hidden, weight, t_ids, lens, out, h = _setup(w, 896, device_gen=True)
    _check_fwd(w, out, h)
    dh, dw, ws = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"])
    assert n.grpo_check_error(ws) == 0
    rng = np.random.default_rng(5)
    L = h["len"]
    rows = []
    for _ in range(24):
        i = int(rng.integers(0, w.N))
        rows.append((i, int(rng.integers(0, L[i]))))
    rows += [(0, 0), (w.N - 1, int(L[-1]) - 1)]
    targets = [int(h["ids"][i, w.P + t]) for i, t in rows[:16]]
    vocab = sorted(set(targets) | set(rng.integers(0, w.V, 24).tolist()) | {0, w.V - 1})
    gr = oracle.lmhead_grads(h["Hn"], h["Wn"], w.P, w.C, h["ids"], L, h["lse"], h["w"], 1.0,
                             rows=rows, vocab=vocab, magnitudes=True)
    dh_h = dh.cpu().numpy()
    got = np.stack([dh_h[i, w.P - 1 + t] for i, t in rows])
    assert_grad(got, gr["dhidden"], gr["dhidden_mag"], "dhidden rows")
    assert_grad(dw.cpu().numpy()[vocab], gr["dweight"], gr["dweight_mag"], "dweight rows")
    scored = np.zeros((w.N, w.T), bool)
    for i in range(w.N):
        scored[i, w.P - 1:w.P - 1 + L[i]] = True
    assert not dh_h[~scored].any()
    assert np.isfinite(dh_h).all() and torch.isfinite(dw).all()


def test_lmhead_grads_sampled_kl_workload():
    """The k3-KL workload's shapes (B=1, G=16, P=256, C=512, V = 151,936,
    about 6,000 scored rows: 24 row blocks, many vocabulary splits of dhidden,
    95 k-steps per dweight item) with hidden size 896: the forward against the
    oracle on every token; sampled dhidden rows and dweight rows (targets of
    scored tokens among them) element by element."""
    n = H.g()
    w = H.with_contrast(wl.QWEN_G16_KL)
    hidden, weight, t_ids, lens, out, h = _setup(w, 896, device_gen=True)
    _check_fwd(w, out, h)
    two = torch.tensor([2.0], dtype=torch.float32, device="cuda")
    dh, dw, ws = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                                        two)
    assert n.grpo_check_error(ws) == 0
    rng = np.random.default_rng(11)
    L = h["len"]
    rows = []
    for _ in range(20):
        i = int(rng.integers(0, w.N))
        rows.append((i, int(rng.integers(0, L[i]))))
    rows += [(w.N - 1, int(L[-1]) - 1)]
    targets = [int(h["ids"][i, w.P + t]) for i, t in rows[:12]]
    vocab = sorted(set(targets) | set(rng.integers(0, w.V, 20).tolist()) | {w.V - 1})
    gr = oracle.lmhead_grads(h["Hn"], h["Wn"], w.P, w.C, h["ids"], L, h["lse"], h["w"], 2.0,
                             rows=rows, vocab=vocab, magnitudes=True)
    dh_h = dh.cpu().numpy()
    got = np.stack([dh_h[i, w.P - 1 + t] for i, t in rows])
    assert_grad(got, gr["dhidden"], gr["dhidden_mag"], "dhidden rows")
    assert_grad(dw.cpu().numpy()[vocab], gr["dweight"], gr["dweight_mag"], "dweight rows")
    scored = np.zeros((w.N, w.T), bool)
    for i in range(w.N):
        scored[i, w.P - 1:w.P - 1 + L[i]] = True
    assert not dh_h[~scored].any()


def test_lmhead_grads_skip_zero_weight():
    """GRPO_BWD_SKIP_ZERO_WEIGHT: two groups, one without reward contrast
    (beta = 0, so its tokens' weights are exactly 0): the same gradients as
    without the flag (dhidden bit for bit on the rows that carry weight, +0 on
    the skipped ones; dweight to float rounding), both against the oracle;
    with every weight 0 both gradients are exactly 0."""
    n = H.g()
    w = wl.variant(wl.QWEN_G8, name="lmg_skip", B=2, G=4, P=6, C=30, V=2000, eos_id=1999,
                   seed=95, forced={"rewards": [1, 0, 0, 1, 0, 0, 0, 0]})
    hidden, weight, t_ids, lens, out, h = _setup(w, 256)
    _check_fwd(w, out, h)
    assert np.all(h["w"][4:] == 0) and np.any(h["w"][:4] != 0)
    a = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"])
    b = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"], flags=1)
    assert n.grpo_check_error(b[2]) == 0
    gr = oracle.lmhead_grads(h["Hn"], h["Wn"], w.P, w.C, h["ids"], h["len"], h["lse"], h["w"],
                             1.0, magnitudes=True)
    for dh, dw in (a[:2], b[:2]):
        assert_grad(dh.cpu().numpy(), gr["dhidden"], gr["dhidden_mag"], "dhidden")
        assert_grad(dw.cpu().numpy(), gr["dweight"], gr["dweight_mag"], "dweight")
    assert torch.equal(a[0][:4], b[0][:4])
    assert not b[0][4:].any()
    assert torch.equal(b[0][4:].view(torch.int32), torch.zeros_like(b[0][4:]).view(torch.int32))
    zero_w = torch.zeros_like(out["w"])
    c = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], zero_w, flags=1)
    torch.cuda.synchronize()
    assert not c[0].any() and not c[1].any()


def test_lmhead_loss_seq_mean_and_its_gradients():
    """grpo_lmhead_loss_fwd_ex with the per-response mean (the original GRPO
    aggregation): loss and w against the oracle's seq-mean loss, and the
    backward with those weights against the oracle's gradients."""
    n = H.g()
    w = H.with_contrast(wl.variant(wl.QWEN_G16_KL, name="lmg_seqmean", B=1, G=4, P=5, C=24,
                                   V=1500, eos_id=1499, seed=97))
    d = 128
    hidden = wl.make_hidden(w, d, "cpu").cuda()
    weight = wl.make_lm_head(w, d, "cpu").cuda()
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    Hn, Wn = _bits16(hidden), _bits16(weight)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage(R, w.G)
    lp_o, lse_o = oracle.lmhead_logp(Hn, Wn, w.P, w.C, ids, len_o)
    old, ref = H.host_inputs(w, lp_o, m_o)
    kinks = np.array([-np.log1p(w.eps), -np.log1p(-w.eps)])
    with np.errstate(invalid="ignore"):
        dist = np.min(np.abs((old.astype(np.float64) - lp_o)[..., None] - kinks), axis=-1)
        old[dist < 1e-3] += np.float32(2e-3)
    loss_o, w_o, ell_o = oracle.loss_seq_mean(lp_o, old.astype(np.float64),
                                              ref.astype(np.float64), A_o, len_o, w.eps, w.beta)
    t_ids = H.dev(ids)
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(R), w.G)
    out = n.grpo_lmhead_loss_fwd(hidden, weight, w.P, t_ids, lens, adv, H.dev(old), H.dev(ref),
                                 w.eps, w.beta, agg=n.GRPO_AGG_SEQ_MEAN)
    assert n.grpo_check_error(out["workspace"]) == 0
    H.assert_loss(float(out["loss"].item()), loss_o, ell_o, float(w.N))
    wt = out["w"].cpu().numpy().astype(np.float64)
    ok = m_o == 1
    # the size of w's two terms, per token: (|A| r + beta (1 + exp(ref - logp))) / (N len_i)
    scale = H.w_scale(lp_o, old, ref, A_o, w.beta, 1.0) / (w.N * np.maximum(len_o, 1)[:, None])
    assert np.all(np.abs(wt - w_o)[ok] <= 1e-4 * scale[ok] + 1e-12)
    dh, dw, ws = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"])
    gr = oracle.lmhead_grads(Hn, Wn, w.P, w.C, ids, len_o, lse_o, w_o, 1.0, magnitudes=True)
    assert_grad(dh.cpu().numpy(), gr["dhidden"], gr["dhidden_mag"], "dhidden")
    assert_grad(dw.cpu().numpy(), gr["dweight"], gr["dweight_mag"], "dweight")


PASSES = wl.variant(wl.QWEN_G16_KL, name="lmg_passes", B=2, G=8, P=5, C=100, V=4099,
                    eos_id=4000, seed=84)
# beta = 0 and a second group without reward contrast: with the skip flag its
# rows (every weight 0) take no part, so the passes hold only group 0's rows
PASSES_SKIP = wl.variant(PASSES, name="lmg_passes_skip", beta=0.0, ref_sigma=None,
                         forced={"rewards": [1.0, 0.0, 0.0, 1.0, 0.0, 1.0, 0.0, 0.0] + [0.0] * 8})


# two 512-column d tiles (896 = 512 + 384) and 40 vocabulary blocks: 80
# dweight items per pass, more than one round of CTA pairs, so every pass adds
# its items with the d tiles rotated over the rounds
PASSES_WIDE = wl.variant(PASSES, name="lmg_passes_wide", V=10007, eos_id=10000)


@pytest.mark.parametrize("rows_per_pass,flags,wk,d",
                         [(256, None, PASSES, 384), (512, None, PASSES, 384),
                          (256, 1, PASSES_SKIP, 384), (0, 1, PASSES_SKIP, 384),
                          (256, None, PASSES_WIDE, 896)],
                         ids=["R256", "R512", "R256_skip", "one_pass_skip", "R256_d896"])
def test_lmhead_grads_in_passes(rows_per_pass, flags, wk, d):
    """The backward in passes of 256 or 512 rows (several passes with rows,
    a ragged last one, and passes with none) against the oracle element by
    element: each pass stores or adds its part of dweight and writes its rows
    of dhidden."""
    n = H.g()
    w = H.with_contrast(wk)
    hidden, weight, t_ids, lens, out, h = _setup(w, d)
    T_valid = int(h["len"].sum())
    assert T_valid > 2 * 256 + 1 and T_valid % 256 != 0
    g = 2.5
    gt = torch.tensor([g], dtype=torch.float32, device="cuda")
    need = n.grpo_lmhead_bwd_workspace_size(w.N, w.C, w.V, d, rows_per_pass)
    full = n.grpo_lmhead_bwd_workspace_size(w.N, w.C, w.V, d)
    assert (need < full) == (rows_per_pass > 0)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    dh, dw, _ = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                                       gt, workspace=ws, flags=flags)
    assert n.grpo_check_error(ws) == 0
    gr = oracle.lmhead_grads(h["Hn"], h["Wn"], w.P, w.C, h["ids"], h["len"], h["lse"], h["w"], g,
                             magnitudes=True)
    assert_grad(dh.cpu().numpy(), gr["dhidden"], gr["dhidden_mag"], "dhidden")
    assert_grad(dw.cpu().numpy(), gr["dweight"], gr["dweight_mag"], "dweight")
    # a second call on the same workspace gives the same bits (dweight is
    # stored again by the first pass, not added to the last call's)
    dh2, dw2, _ = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                                         gt, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(dh.view(torch.int32), dh2.view(torch.int32))
    assert torch.equal(dw.view(torch.int32), dw2.view(torch.int32))


def test_lmhead_grads_workspace_by_scored_rows():
    """A workspace sized for the scored rows actually present (their count
    rounded up to 256) runs one pass with rows; one smaller than a single
    256-row pass is refused."""
    n = H.g()
    w = H.with_contrast(PASSES)
    hidden, weight, t_ids, lens, out, h = _setup(w, 384)
    T_valid = int(h["len"].sum())
    ws = torch.empty((n.grpo_lmhead_bwd_workspace_size(w.N, w.C, w.V, 384, T_valid),),
                     dtype=torch.uint8, device="cuda")
    a = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                               workspace=ws)
    b = n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"])
    torch.cuda.synchronize()
    # the same single pass over the scored rows: the same bits as the
    # workspace for every possible row
    assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    small = torch.empty((n.grpo_lmhead_bwd_workspace_size(w.N, w.C, w.V, 384, 256) - 1,),
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(n.GrpoError):
        n.grpo_lmhead_loss_bwd(hidden, weight, w.P, t_ids, lens, out["lse"], out["w"],
                               workspace=small)
