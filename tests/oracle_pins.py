"""Pins for the float64 CPU oracle: checks against things other than the oracle.

Each ``pin_*`` function takes a loaded :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with what the pages or the
mathematics fix: values the pages print, hand-derived cases from the pages'
definitions (``tests/golden/``), closed forms, library routines (scipy), and
central finite differences.  ``test_oracle_pins.py`` runs them against the
real oracle; ``test_oracle_mutants.py`` runs them against builds with planted
mistakes and requires each mistake to fail at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np

from vocab_wide_logprob_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(fname):
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line


# --------------------------------------------------------------------------
# "The completion mask"
# --------------------------------------------------------------------------

def mask_cases():
    cases = []
    for line in _rows("mask_cases.txt"):
        eos, prompt, comp, exp_mask, exp_len = [s.split() for s in line.split("|")]
        cases.append((int(eos[0]), [int(x) for x in prompt], [int(x) for x in comp],
                      [int(x) for x in exp_mask], int(exp_len[0])))
    return cases


def pin_mask_golden(o):
    for eos, prompt, comp, exp_mask, exp_len in mask_cases():
        ids = np.array([prompt + comp], np.int64)
        m, ln = o.mask(ids, len(prompt), len(comp), eos)
        assert m[0].tolist() == exp_mask, (prompt, comp, m[0].tolist(), exp_mask)
        assert int(ln[0]) == exp_len, (prompt, comp, int(ln[0]), exp_len)


def pin_mask_batch_matches_rows(o):
    """All golden cases with equal shapes stacked into one batch give the
    same rows as one at a time (no cross-row leakage)."""
    cases = [c for c in mask_cases() if len(c[1]) == 2 and len(c[2]) == 6 and c[0] == 2]
    ids = np.array([c[1] + c[2] for c in cases], np.int64)
    m, ln = o.mask(ids, 2, 6, 2)
    assert m.tolist() == [c[3] for c in cases]
    assert ln.tolist() == [c[4] for c in cases]


# --------------------------------------------------------------------------
# "Dr. GRPO" advantage: A_i = R_i - mean of the group, no sigma
# --------------------------------------------------------------------------

def pin_advantage_examples(o):
    # hand-derived: one success among four -> mean 1/4
    assert o.advantage(np.array([1, 0, 0, 0.]), 4).tolist() == [0.75, -0.25, -0.25, -0.25]
    # two groups of four: (1,1,0,0) mean 1/2; (0,0,0,1) mean 1/4
    assert o.advantage(np.array([1, 1, 0, 0, 0, 0, 0, 1.]), 4).tolist() == \
        [0.5, 0.5, -0.5, -0.5, -0.25, -0.25, -0.25, 0.75]
    # uniform groups carry no contrast: every advantage is exactly zero
    assert o.advantage(np.ones(8), 8).tolist() == [0.0] * 8
    assert o.advantage(np.zeros(16), 16).tolist() == [0.0] * 16
    # no division by the group's standard deviation: scaling rewards by 3
    # scales advantages by 3 (a sigma-normalised advantage would not change)
    a1 = o.advantage(np.array([1, 0, 0, 0.]), 4)
    a3 = o.advantage(np.array([3, 0, 0, 0.]), 4)
    assert np.allclose(a3, 3 * a1, rtol=0, atol=1e-15)
    # G = 3, real rewards: mean 0.5 -> (0.5, -0.25, -0.25)
    assert np.allclose(o.advantage(np.array([1.0, 0.25, 0.25]), 3), [0.5, -0.25, -0.25],
                       rtol=0, atol=1e-15)
    # G = 1: a single completion is its own baseline
    assert o.advantage(np.array([1.0, 0.0]), 1).tolist() == [0.0, 0.0]


def no_contrast_golden():
    out = []
    for line in _rows("no_contrast.txt"):
        q, p, G, printed, dec = line.split()
        out.append((q, float(p), int(G), float(printed), int(dec)))
    return out


def pin_printed_probabilities():
    """The closed forms reproduce the digits the pages print."""
    for q, p, G, printed, dec in no_contrast_golden():
        val = (1 - p) ** G if q == "all_fail" else (1 - p) ** G + p ** G
        assert round(val, dec) == printed, (q, p, G, val, printed)


def pin_advantage_monte_carlo(o, groups=1_000_000):
    """Rewards from the generator's Bernoulli draw, advantages from the
    oracle: the fraction of groups whose advantages are all zero matches the
    pages' closed form (1-p)^G + p^G within 4 standard errors, and the mixture
    p ~ U(0, 1/2) used by the batched workload matches its closed form 2/9."""
    cases = [(0.05, 8, 0.95 ** 8 + 0.05 ** 8), (0.05, 16, 0.95 ** 16 + 0.05 ** 16)]
    for p, G, exact in cases:
        w = wl.Workload("mc", B=groups, G=G, P=1, C=1, V=2, dtype="f32", logit_std=1.0,
                        eos_id=0, reward_p=p, seed=777 + G)
        A = o.advantage(wl.make_rewards(w), G).reshape(groups, G)
        frac = float(np.mean(np.all(A == 0.0, axis=1)))
        se = math.sqrt(exact * (1 - exact) / groups)
        assert abs(frac - exact) < 4 * se, (p, G, frac, exact, se)
    # int_0^{1/2} [(1-p)^8 + p^8] dp / (1/2) = 2 * (1/9) = 2/9 for G = 8
    w = wl.Workload("mc_mix", B=groups, G=8, P=1, C=1, V=2, dtype="f32", logit_std=1.0,
                    eos_id=0, reward_p_range=(0.0, 0.5), seed=4242)
    A = o.advantage(wl.make_rewards(w), 8).reshape(groups, 8)
    frac = float(np.mean(np.all(A == 0.0, axis=1)))
    exact = 2.0 / 9.0
    se = math.sqrt(exact * (1 - exact) / groups)
    assert abs(frac - exact) < 4 * se, (frac, exact, se)


# --------------------------------------------------------------------------
# reward contrast ("The Quiet Library", "The sparse-reward bottleneck"): a
# group whose rewards are all equal has no contrast; the others are useful
# --------------------------------------------------------------------------

def pin_contrast_count_examples(o):
    """Hand-counted groups: the differing reward may sit first, in the middle
    or last in its group; G = 1 never has contrast; real-valued rewards."""
    cases = [
        ([1, 0, 0, 0], 4, 1),
        ([0, 0, 0, 1], 4, 1),               # only the last reward differs
        ([0, 0, 1, 0], 4, 1),
        ([1, 1, 1, 1, 0, 0, 0, 0], 4, 0),   # two uniform groups (all pass, all fail)
        ([0, 0, 0, 1, 1, 1, 1, 1, 0, 1, 0, 0], 4, 2),
        ([1, 1, 0, 0, 0, 0, 0, 0], 4, 1),   # group 1 equals group 0's last rewards
        ([1, 0, 1, 0, 1, 1], 2, 2),
        ([1.0, 0.0, 1.0], 1, 0),            # a single completion is never contrasted
        ([0.5, 0.5, 0.5, 0.5, 0.5, 0.25], 3, 1),
        ([], 4, 0),
    ]
    for R, G, want in cases:
        got = o.contrast_count(np.array(R, np.float64), G)
        assert got == want, (R, G, got, want)


def pin_contrast_count_monte_carlo(o, groups=200_000):
    """Binary rewards from the generator's Bernoulli draw: the fraction of
    groups the oracle counts as contrasted is 1 - [(1-p)^G + p^G], the
    complement of the pages' no-contrast probability (0.6634 printed at
    p = 0.05, G = 8; 0.4401 all-fail at G = 16), within 4 standard errors."""
    printed = {(p, G): v for q, p, G, v, _ in no_contrast_golden() if q == "no_contrast"}
    for p, G in ((0.05, 8), (0.05, 16), (0.3, 4)):
        exact = (1 - p) ** G + p ** G
        if (p, G) in printed:
            assert abs(exact - printed[(p, G)]) < 1e-4
        w = wl.Workload("mc_c", B=groups, G=G, P=1, C=1, V=2, dtype="f32", logit_std=1.0,
                        eos_id=0, reward_p=p, seed=991 + G)
        frac = o.contrast_count(wl.make_rewards(w), G) / groups
        se = math.sqrt(exact * (1 - exact) / groups)
        assert abs(frac - (1 - exact)) < 4 * se, (p, G, frac, 1 - exact, se)


# --------------------------------------------------------------------------
# "compute_logprobs": shift by one, log_softmax, gather
# --------------------------------------------------------------------------

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_logp_constant_row(o):
    """A constant row is the uniform distribution: logp = -ln V exactly."""
    for V in (1, 7, 1024, 151936):
        for c in (0.0, 3.7, -120.5):
            row = np.full((1, V), c, np.float64)
            lp, ls = o.logp_rows(row, "f64", np.array([V // 2]))
            assert abs(lp[0] + math.log(V)) <= 1e-12 * max(1.0, math.log(V)), (V, c, lp)
            assert abs(ls[0] - (c + math.log(V))) <= 1e-12 * max(1.0, abs(c) + 12), (V, c, ls)


def pin_logp_two_level(o):
    """k entries equal to a, the rest equal to b: closed-form logsumexp
    a + ln(k + (V-k) e^(b-a))."""
    for V, k, a, b in [(1024, 1, 9.0, 0.0), (151936, 5, 2.5, -1.0), (33, 32, 0.0, 4.0)]:
        row = np.full(V, b, np.float64)
        row[:k] = a
        lse = a + math.log(k + (V - k) * math.exp(b - a))
        lp, ls = o.logp_rows(row[None, :], "f64", np.array([0]))
        assert abs(ls[0] - lse) < 1e-12 * max(1, abs(lse)), (V, k, ls[0], lse)
        assert abs(lp[0] - (a - lse)) < 1e-12 * max(1, abs(lse)), (V, k, lp[0], a - lse)
        lp2, _ = o.logp_rows(row[None, :], "f64", np.array([V - 1]))
        assert abs(lp2[0] - (b - lse)) < 1e-12 * max(1, abs(lse))


def pin_logp_library(o):
    """Random rows in f64, f32 and bf16 against scipy.special.log_softmax."""
    from scipy.special import log_softmax
    rng = np.random.default_rng(5)
    for V in (2, 1000, 1003, 151936):
        x = rng.normal(0.0, 3.0, size=(4, V))
        y = rng.integers(0, V, size=4)
        ref = log_softmax(x, axis=1)[np.arange(4), y]
        lp, _ = o.logp_rows(x, "f64", y)
        assert np.max(np.abs(lp - ref)) < 1e-11, (V, np.max(np.abs(lp - ref)))
        x32 = x.astype(np.float32)
        ref32 = log_softmax(x32.astype(np.float64), axis=1)[np.arange(4), y]
        lp32, _ = o.logp_rows(x32, "f32", y)
        assert np.max(np.abs(lp32 - ref32)) < 1e-11
        xb = _bf16_bits(x32)
        refb = log_softmax(_bf16_to_f64(xb), axis=1)[np.arange(4), y]
        lpb, _ = o.logp_rows(xb, "bf16", y)
        assert np.max(np.abs(lpb - refb)) < 1e-11
    # rows with -inf entries (a masked vocabulary) and a huge spread
    x = np.array([[-np.inf, 0.0, 1.0, -np.inf, 80.0, -80.0]])
    ref = log_softmax(x, axis=1)
    for y in (1, 2, 4, 5):
        lp, _ = o.logp_rows(x, "f64", np.array([y]))
        assert abs(lp[0] - ref[0, y]) < 1e-12, (y, lp[0], ref[0, y])
    lp, _ = o.logp_rows(x, "f64", np.array([0]))
    assert lp[0] == -np.inf


def pin_logp_token_range(o):
    """A sampled id outside [0, V) is refused."""
    for bad in (-1, 8):
        try:
            o.logp_rows(np.zeros((1, 8)), "f64", np.array([bad]))
        except ValueError:
            continue
        raise AssertionError(f"token id {bad} accepted")


def pin_logp_shift(o):
    """"logits at position t predict the token at t+1": completion token t is
    scored by logits row P-1+t.  Plant a large logit at (row P-1+t, column
    y_t) for even t only; rows of odd t stay all-zero.  Then logp is ~0 at
    even t and exactly -ln V at odd t; a shift by one swaps the pattern."""
    N, P, C, V, big = 3, 5, 8, 64, 60.0
    rng = np.random.default_rng(11)
    ids = rng.integers(3, V, size=(N, P + C))
    lens = np.array([C, 5, 1], np.int32)
    z = np.zeros((N, P + C, V))
    for i in range(N):
        for t in range(0, C, 2):
            z[i, P - 1 + t, ids[i, P + t]] = big
    lp, ls = o.logp(z, "f64", P, C, ids, lens)
    for i in range(N):
        for t in range(C):
            if t >= lens[i]:
                assert lp[i, t] == 0.0 and ls[i, t] == 0.0
            elif t % 2 == 0:
                assert -1e-20 < lp[i, t] <= 0.0 and lp[i, t] > -(V) * math.exp(-big) * 1.01
            else:
                assert abs(lp[i, t] + math.log(V)) < 1e-12, (i, t, lp[i, t])


# --------------------------------------------------------------------------
# "The loss": clipped surrogate, KL, token-sum / constant
# --------------------------------------------------------------------------

def surrogate_cases():
    return [tuple(float(x) for x in line.split()) for line in _rows("surrogate_cases.txt")]


def kl_cases():
    return [tuple(float(x) for x in line.split()) for line in _rows("kl_cases.txt")]


def pin_surrogate_golden(o):
    """One token per completion, norm 1, beta 0: ell = -s, w = -ds."""
    for A, r, eps, s, ds in surrogate_cases():
        lp = np.array([[-2.0]])
        old = lp - math.log(r)   # exp(lp - old) = r
        loss, w, ell = o.loss(lp, old, None, np.array([A]), np.array([1], np.int32),
                              eps, 0.0, 1.0)
        assert abs(ell[0, 0] + s) < 1e-12, (A, r, eps, ell[0, 0], -s)
        assert abs(loss + s) < 1e-12
        assert abs(w[0, 0] + ds) < 1e-12, (A, r, eps, w[0, 0], -ds)


def pin_kl_golden(o):
    """Zero advantage, beta 0.5, norm 2: ell = beta*k3, w = beta*dk3/norm."""
    beta, norm = 0.5, 2.0
    for d, k3, dk3 in kl_cases():
        lp = np.array([[-1.25]])
        ref = lp + d
        loss, w, ell = o.loss(lp, None, ref, np.array([0.0]), np.array([1], np.int32),
                              0.2, beta, norm)
        assert abs(ell[0, 0] - beta * k3) < 1e-14, (d, ell[0, 0], beta * k3)
        assert abs(loss - beta * k3 / norm) < 1e-14
        assert abs(w[0, 0] - beta * dk3 / norm) < 1e-14, (d, w[0, 0], beta * dk3 / norm)


def _tiny_inputs(o):
    w = wl.TINY
    ids = wl.make_ids(w)
    z, dt = wl.logits_as_numpy(wl.make_logits_cpu(w))
    m, lens = o.mask(ids, w.P, w.C, w.eos_id)
    A = o.advantage(wl.make_rewards(w), w.G)
    lp, ls = o.logp(z, dt, w.P, w.C, ids, lens)
    return w, ids, z, dt, m, lens, A, lp, ls


def pin_step0_identity(o):
    """"On inner step 0 ... ratio is exactly 1 everywhere and the loss reduces
    to -(advantages * mask).sum(dim=1).mean()": with the constant N*C the same
    identity reads loss = -sum_i A_i len_i / (N*C); with norm = N it is the
    page's own expression."""
    w, ids, z, dt, m, lens, A, lp, ls = _tiny_inputs(o)
    N, C = w.N, w.C
    page_value = -float(np.mean(np.sum(A[:, None] * m, axis=1)))
    for old in (None, lp.copy()):
        loss, wt, ell = o.loss(lp, old, None, A, lens, w.eps, 0.0)
        assert abs(loss - page_value * N / (N * C)) < 1e-14, (loss, page_value / C)
        loss_n, _, _ = o.loss(lp, old, None, A, lens, w.eps, 0.0, float(N))
        assert abs(loss_n - page_value) < 1e-13, (loss_n, page_value)
        assert np.allclose(wt, -(A[:, None] * m) / (N * C), rtol=0, atol=1e-17)
    # zero advantages and no KL: no loss and no gradient at all
    loss, wt, _ = o.loss(lp, None, None, np.zeros(N), lens, w.eps, 0.0)
    assert loss == 0.0 and not np.any(wt)


def pin_ratio_closed_form(o):
    """old = logp - ln r0 on every token gives r = r0; for r0 = 1.5, eps 0.2 the
    surrogate is 1.2*A for A > 0 and 1.5*A for A < 0."""
    w, ids, z, dt, m, lens, A, lp, ls = _tiny_inputs(o)
    N, C = w.N, w.C
    old = lp - math.log(1.5)
    s = np.where(A > 0, 1.2 * A, 1.5 * A)
    expect = -float(np.sum(s * lens)) / (N * C)
    loss, wt, ell = o.loss(lp, old, None, A, lens, 0.2, 0.0)
    assert abs(loss - expect) < 1e-13, (loss, expect)
    ds = np.where(A > 0, 0.0, 1.5 * A)
    assert np.allclose(wt, -(ds[:, None] * m) / (N * C), rtol=0, atol=1e-15)


def pin_kl_closed_form(o):
    """Uniform rewards (A = 0), ref = logp + ln 2: every valid token adds
    beta*(1 - ln 2), and w = -beta/(N*C) on valid tokens."""
    w, ids, z, dt, m, lens, A, lp, ls = _tiny_inputs(o)
    N, C = w.N, w.C
    beta = 0.04
    ref = lp + math.log(2.0)
    loss, wt, _ = o.loss(lp, None, ref, np.zeros(N), lens, 0.2, beta)
    expect = beta * (1 - math.log(2.0)) * float(lens.sum()) / (N * C)
    assert abs(loss - expect) < 1e-15, (loss, expect)
    assert np.allclose(wt, -beta * m / (N * C), rtol=0, atol=1e-17)


def pin_masked_never_read(o):
    """Old and reference log-probs past the first EOS are padding: NaN there
    changes nothing ("the mask multiplies per_token_loss, not ratio")."""
    w, ids, z, dt, m, lens, A, lp, ls = _tiny_inputs(o)
    rng = np.random.default_rng(3)
    old = lp + rng.normal(0, 0.1, lp.shape)
    ref = lp + rng.normal(0, 0.1, lp.shape)
    l1, w1, e1 = o.loss(lp, old, ref, A, lens, 0.2, 0.04)
    old[m == 0] = np.nan
    ref[m == 0] = np.nan
    l2, w2, e2 = o.loss(lp, old, ref, A, lens, 0.2, 0.04)
    assert l1 == l2 and np.array_equal(w1, w2) and np.array_equal(e1, e2)
    assert np.all(e2[m == 0] == 0.0) and np.all(w2[m == 0] == 0.0)


# --------------------------------------------------------------------------
# "loss.backward()": gradient with respect to the logits
# --------------------------------------------------------------------------

def _away_from_kinks(rng, shape, eps):
    """Noise on log-probs whose ratio exp(-noise) stays >= 0.01 (in log space)
    away from the clip boundaries 1-eps and 1+eps."""
    kinks = np.array([-math.log(1 + eps), -math.log(1 - eps)])
    x = rng.normal(0, 0.2, shape)
    bad = np.min(np.abs(x[..., None] - kinks), axis=-1) < 0.01
    x[bad] += 0.05
    return x


def _fd_setup(o, z, P, C, ids, lens, A, eps, beta, norm, seed):
    lp, _ = o.logp(z, "f64", P, C, ids, lens)
    rng = np.random.default_rng(seed)
    old = lp + _away_from_kinks(rng, lp.shape, eps)
    ref = lp + rng.normal(0, 0.3, lp.shape)

    def f(zz):
        lpz, _ = o.logp(zz, "f64", P, C, ids, lens)
        return o.loss(lpz, old, ref, A, lens, eps, beta, norm)[0]

    lp, ls = o.logp(z, "f64", P, C, ids, lens)
    _, wt, _ = o.loss(lp, old, ref, A, lens, eps, beta, norm)
    return f, ls, wt


def _fd_check(o, z, P, C, ids, lens, A, eps, beta, norm, entries, seed, g=1.0):
    f, ls, wt = _fd_setup(o, z, P, C, ids, lens, A, eps, beta, norm, seed)
    an = o.dlogits(z, "f64", P, C, ids, lens, ls, wt, g)
    h = 1e-5
    for (i, r, v) in entries:
        zp = z.copy()
        zp[i, r, v] += h
        zm = z.copy()
        zm[i, r, v] -= h
        fd = g * (f(zp) - f(zm)) / (2 * h)
        a = an[i, r, v]
        assert abs(fd - a) <= 1e-8 + 1e-5 * abs(a), ((i, r, v), fd, a)
    return an


def pin_dlogits_fd_micro(o):
    """Every entry of a micro batch (B=2, G=2, P=2, C=4, V=8) against central
    finite differences of the oracle's own loss (float64 logits, h = 1e-5),
    with clipping, the KL term and masked rows all active."""
    B, G, P, C, V = 2, 2, 2, 4, 8
    rng = np.random.default_rng(21)
    z = rng.normal(0, 2, size=(B * G, P + C, V))
    ids = rng.integers(3, V, size=(B * G, P + C))
    ids[1, P + 2] = 2          # EOS at index 2 -> length 3
    ids[2, P + 0:] = 2         # EOS first -> length 1
    _, lens = o.mask(ids, P, C, 2)
    assert lens.tolist() == [4, 3, 1, 4]
    A = o.advantage(np.array([1, 0, 0, 1.]), G)
    entries = [(i, r, v) for i in range(B * G) for r in range(P + C) for v in range(V)]
    an = _fd_check(o, z, P, C, ids, lens, A, 0.2, 0.1, 1.0, entries, seed=22)
    # invariants: each scored row sums to zero; rows that score nothing are 0
    for i in range(B * G):
        for r in range(P + C):
            t = r - (P - 1)
            if 0 <= t < lens[i]:
                assert abs(an[i, r].sum()) < 1e-14
            else:
                assert not np.any(an[i, r])


def pin_dlogits_fd_tiny(o):
    """200 random entries of the tiny workload (logits widened to float64),
    half of them in scored rows, with old/ref noise, beta = 0.04, norm 1,
    and an upstream gradient g = 2.5."""
    w, ids, z, dt, m, lens, A, lp, ls = _tiny_inputs(o)
    z = z.astype(np.float64)
    rng = np.random.default_rng(23)
    entries = []
    for _ in range(100):
        i = int(rng.integers(0, w.N))
        t = int(rng.integers(0, lens[i]))
        v = int(ids[i, w.P + t]) if rng.random() < 0.3 else int(rng.integers(0, w.V))
        entries.append((i, w.P - 1 + t, v))
    for _ in range(100):
        entries.append((int(rng.integers(0, w.N)), int(rng.integers(0, w.T)),
                        int(rng.integers(0, w.V))))
    _fd_check(o, z, w.P, w.C, ids, lens, A, 0.2, 0.04, 1.0, entries, seed=24, g=2.5)


def pin_dlogits_row_closed_form(o):
    """Constant row (uniform softmax 1/V): out = gw*(onehot - 1/V)."""
    V, y, gw = 16, 5, 0.3
    row = np.zeros(V)
    out = o.dlogits_row(row, "f64", y, math.log(V), gw)
    expect = np.full(V, -gw / V)
    expect[y] += gw
    assert np.allclose(out, expect, rtol=0, atol=1e-16)


# --------------------------------------------------------------------------
# original GRPO options: sigma-normalised advantage, per-response mean
# --------------------------------------------------------------------------

def pin_advantage_std_examples(o):
    """Section "GRPO": A_i = (R_i - mu)/sigma inside the group.  One success
    among four: mu = 1/4, sigma = sqrt(3)/4, so A = (sqrt 3, -1/sqrt 3, ...);
    in general a success scores sqrt((1-p)/p) for p = k/G.  The advantage is
    unchanged by scaling or shifting the rewards (the "difficulty bias" the
    page attributes to dividing by sigma)."""
    s3 = math.sqrt(3.0)
    A = o.advantage_std(np.array([1, 0, 0, 0.]), 4)
    assert np.allclose(A, [s3, -1 / s3, -1 / s3, -1 / s3], rtol=0, atol=1e-15), A
    for k, G in [(1, 8), (3, 8), (5, 16)]:
        R = np.zeros(G)
        R[:k] = 1
        p = k / G
        A = o.advantage_std(R, G)
        assert abs(A[0] - math.sqrt((1 - p) / p)) < 1e-14 and abs(A[-1] + math.sqrt(p / (1 - p))) < 1e-14
    R = np.array([0.3, 1.7, -2.0, 0.5, 4.0, 4.0, 0.0, 1.0])
    base = o.advantage_std(R, 4)
    assert np.allclose(o.advantage_std(3 * R + 5, 4), base, rtol=0, atol=1e-13)
    assert np.allclose(base.reshape(2, 4).sum(1), 0.0, atol=1e-13)
    assert np.allclose((base.reshape(2, 4) ** 2).mean(1), 1.0, atol=1e-13)  # unit variance
    # a uniform group: 0 / (0 + std_eps) = 0
    assert o.advantage_std(np.ones(4), 4, 1e-4).tolist() == [0.0] * 4


def pin_seq_mean_aggregation(o):
    """Section "Dr. GRPO": the original loss averages per response by 1/|o_i|.
    Two completions of lengths 2 and 4, ratio 1, A = (0.5, -0.5): every token's
    loss is -A_i, so loss = ((-0.5*2)/2 + (0.5*4)/4) / 2 = 0, and
    w = -A_i / (N * len_i) = (-0.125, 0.0625)."""
    lp = np.full((2, 4), -3.0)
    lens = np.array([2, 4], np.int32)
    loss, w, ell = o.loss_seq_mean(lp, None, None, np.array([0.5, -0.5]), lens, 0.2, 0.0)
    assert abs(loss) < 1e-15, loss
    assert np.allclose(w, [[-0.125, -0.125, 0, 0], [0.0625] * 4], rtol=0, atol=1e-16), w
    # lengths no longer weight the loss: doubling one response's length with
    # the same per-token loss leaves its contribution unchanged
    A = np.array([1.0, 1.0])
    l1, _, _ = o.loss_seq_mean(lp, None, None, A, np.array([1, 2], np.int32), 0.2, 0.0)
    l2, _, _ = o.loss_seq_mean(lp, None, None, A, np.array([2, 4], np.int32), 0.2, 0.0)
    assert abs(l1 - l2) < 1e-15 and abs(l1 + 1.0) < 1e-15
    # with equal lengths L it equals the token sum over the constant N*L
    w0 = wl.TINY
    ids = wl.make_ids(w0)
    _, ln = o.mask(ids, w0.P, w0.C, w0.eos_id)
    L = np.full_like(ln, 7)
    rng = np.random.default_rng(8)
    lpr = rng.normal(-5, 1, size=(w0.N, w0.C))
    old = lpr + rng.normal(0, 0.2, size=lpr.shape)
    Ar = rng.normal(0, 1, size=w0.N)
    a, wa, _ = o.loss_seq_mean(lpr, old, None, Ar, L, 0.2, 0.0)
    b, wb, _ = o.loss(lpr, old, None, Ar, L, 0.2, 0.0, float(w0.N * 7))
    assert abs(a - b) < 1e-14 and np.allclose(wa, wb, rtol=0, atol=1e-16)


def pin_dlogits_fd_seq_mean(o):
    """Finite differences of the per-response-mean loss on the micro batch."""
    B, G, P, C, V = 2, 2, 2, 4, 8
    rng = np.random.default_rng(31)
    z = rng.normal(0, 2, size=(B * G, P + C, V))
    ids = rng.integers(3, V, size=(B * G, P + C))
    ids[1, P + 2] = 2
    _, lens = o.mask(ids, P, C, 2)
    A = o.advantage_std(np.array([1, 0, 0, 1.]), G, 1e-4)
    lp, _ = o.logp(z, "f64", P, C, ids, lens)
    old = lp + _away_from_kinks(rng, lp.shape, 0.2)
    ref = lp + rng.normal(0, 0.3, lp.shape)

    def f(zz):
        lpz, _ = o.logp(zz, "f64", P, C, ids, lens)
        return o.loss_seq_mean(lpz, old, ref, A, lens, 0.2, 0.1)[0]

    lp, ls = o.logp(z, "f64", P, C, ids, lens)
    _, wt, _ = o.loss_seq_mean(lp, old, ref, A, lens, 0.2, 0.1)
    an = o.dlogits(z, "f64", P, C, ids, lens, ls, wt)
    h = 1e-5
    for i in range(B * G):
        for r in range(P + C):
            for v in range(0, V, 3):
                zp = z.copy()
                zp[i, r, v] += h
                zm = z.copy()
                zm[i, r, v] -= h
                fd = (f(zp) - f(zm)) / (2 * h)
                assert abs(fd - an[i, r, v]) <= 1e-9 + 1e-5 * abs(an[i, r, v]), (i, r, v)


def pin_lmhead_reduces_to_logits(o):
    """With W = I (d = V) the projection is the identity: the LM-head log-probs
    equal the log-probs of the hidden states taken as logits; permuting W's
    rows permutes the vocabulary, so relabelling the ids gives the same
    log-probs."""
    N, P, C, V = 3, 4, 6, 16
    rng = np.random.default_rng(41)
    H = rng.normal(0, 2, size=(N, P + C, V))
    ids = rng.integers(3, V, size=(N, P + C))
    ids[1, P + 3] = 2
    _, lens = o.mask(ids, P, C, 2)
    a, la = o.lmhead_logp(H, np.eye(V), P, C, ids, lens)
    b, lb = o.logp(H, "f64", P, C, ids, lens)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    perm = rng.permutation(V)
    W = np.eye(V)[perm]            # row v of W picks coordinate perm[v]
    inv = np.argsort(perm)         # token u's logit is coordinate perm[u]...
    ids2 = ids.copy()
    ids2[:, P:] = inv[ids[:, P:]]  # ...so ask for the token whose row is the old one
    c, _ = o.lmhead_logp(H, W, P, C, ids2, lens)
    assert np.allclose(c, b, rtol=0, atol=1e-12)


def _lmhead_micro(o, seed):
    """A micro batch through an LM head: 3 completions (one stops at EOS),
    P=2, C=3, V=7, d=5, float64 hidden states and weights."""
    N, P, C, V, d = 3, 2, 3, 7, 5
    rng = np.random.default_rng(seed)
    H = rng.normal(0, 1, size=(N, P + C, d))
    W = rng.normal(0, 0.8, size=(V, d))
    ids = rng.integers(3, V, size=(N, P + C))
    ids[2, P + 1] = 2                      # completion 2 ends after 2 tokens
    _, lens = o.mask(ids, P, C, 2)
    A = np.array([0.7, -0.3, -0.4])
    lp, _ = o.lmhead_logp(H, W, P, C, ids, lens)
    old = lp + _away_from_kinks(rng, lp.shape, 0.2)
    ref = lp + rng.normal(0, 0.3, lp.shape)
    return H, W, ids, lens, A, old, ref, P, C


def pin_lmhead_grads_fd(o):
    """Chain rule through logits = hidden x W^T: central finite differences of
    the loss as a function of every hidden-state and every weight entry
    (prompt rows, the last row and rows past the EOS included: their
    derivative is 0), with the clipped surrogate and the KL term both active
    and an upstream gradient g = 2.5."""
    H, W, ids, lens, A, old, ref, P, C = _lmhead_micro(o, 51)
    g = 2.5

    def f(HH, WW):
        lpz, _ = o.lmhead_logp(HH, WW, P, C, ids, lens)
        return g * o.loss(lpz, old, ref, A, lens, 0.2, 0.1)[0]

    lp, ls = o.lmhead_logp(H, W, P, C, ids, lens)
    _, wt, _ = o.loss(lp, old, ref, A, lens, 0.2, 0.1)
    an = o.lmhead_grads(H, W, P, C, ids, lens, ls, wt, g)
    h = 1e-6
    for idx in np.ndindex(H.shape):
        Hp = H.copy()
        Hp[idx] += h
        Hm = H.copy()
        Hm[idx] -= h
        fd = (f(Hp, W) - f(Hm, W)) / (2 * h)
        assert abs(fd - an["dhidden"][idx]) <= 1e-9 + 1e-5 * abs(an["dhidden"][idx]), idx
    for idx in np.ndindex(W.shape):
        Wp = W.copy()
        Wp[idx] += h
        Wm = W.copy()
        Wm[idx] -= h
        fd = (f(H, Wp) - f(H, Wm)) / (2 * h)
        assert abs(fd - an["dweight"][idx]) <= 1e-9 + 1e-5 * abs(an["dweight"][idx]), idx


def pin_lmhead_grads_identity_and_subsets(o):
    """With W = I (d = V) the hidden states are the logits, so dhidden equals
    the logits gradient; dweight is then sum over scored rows of dz^T h,
    checked by a plain loop; the row and vocabulary subsets equal the
    matching slices of the full result; the columns of dweight sum to 0
    (each row of dz does), and |value| <= magnitude everywhere."""
    N, P, C, V = 3, 4, 5, 9
    rng = np.random.default_rng(43)
    H = rng.normal(0, 2, size=(N, P + C, V))
    ids = rng.integers(3, V, size=(N, P + C))
    ids[0, P + 1] = 2
    _, lens = o.mask(ids, P, C, 2)
    lp, ls = o.lmhead_logp(H, np.eye(V), P, C, ids, lens)
    old = lp + _away_from_kinks(rng, lp.shape, 0.2)
    _, wt, _ = o.loss(lp, old, None, np.array([1.0, -0.5, -0.5]), lens, 0.2, 0.0)
    gr = o.lmhead_grads(H, np.eye(V), P, C, ids, lens, ls, wt, 1.5, magnitudes=True)
    dz = o.dlogits(H, "f64", P, C, ids, lens, ls, wt, 1.5)
    assert np.allclose(gr["dhidden"], dz, rtol=0, atol=1e-15)
    ref = np.zeros((V, V))
    for i in range(N):
        for t in range(int(lens[i])):
            r = P - 1 + t
            for v in range(V):
                for k in range(V):
                    ref[v, k] += dz[i, r, v] * H[i, r, k]
    assert np.allclose(gr["dweight"], ref, rtol=0, atol=1e-13)
    assert np.all(np.abs(gr["dweight"].sum(axis=0)) < 1e-12)
    assert np.all(np.abs(gr["dhidden"]) <= gr["dhidden_mag"] + 1e-15)
    assert np.all(np.abs(gr["dweight"]) <= gr["dweight_mag"] + 1e-15)
    Hb, Wb, ids_b, lens_b, A, old_b, ref_b, Pb, Cb = _lmhead_micro(o, 52)
    lp, ls = o.lmhead_logp(Hb, Wb, Pb, Cb, ids_b, lens_b)
    _, wt, _ = o.loss(lp, old_b, ref_b, A, lens_b, 0.2, 0.1)
    full = o.lmhead_grads(Hb, Wb, Pb, Cb, ids_b, lens_b, ls, wt)
    rows = [(2, 1), (0, 0), (2, 2), (1, 2)]     # (2, 2) is past completion 2's EOS
    vocab = [6, 0, 3]
    part = o.lmhead_grads(Hb, Wb, Pb, Cb, ids_b, lens_b, ls, wt, rows=rows, vocab=vocab)
    for k, (i, t) in enumerate(rows):
        assert np.allclose(part["dhidden"][k], full["dhidden"][i, Pb - 1 + t], rtol=0, atol=1e-15)
    assert not part["dhidden"][2].any()
    assert np.allclose(part["dweight"], full["dweight"][vocab], rtol=0, atol=1e-15)
    assert not full["dhidden"][:, :Pb - 1].any() and not full["dhidden"][:, -1].any()


ALL_CHEAP = [
    pin_lmhead_reduces_to_logits, pin_lmhead_grads_fd, pin_lmhead_grads_identity_and_subsets,
    pin_advantage_std_examples, pin_seq_mean_aggregation, pin_dlogits_fd_seq_mean,
    pin_mask_golden, pin_mask_batch_matches_rows, pin_advantage_examples,
    pin_contrast_count_examples, pin_contrast_count_monte_carlo,
    pin_logp_constant_row, pin_logp_two_level, pin_logp_library, pin_logp_token_range,
    pin_logp_shift, pin_surrogate_golden, pin_kl_golden, pin_step0_identity,
    pin_ratio_closed_form, pin_kl_closed_form, pin_masked_never_read,
    pin_dlogits_row_closed_form, pin_dlogits_fd_micro, pin_dlogits_fd_tiny,
]
