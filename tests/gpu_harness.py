"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on a seeded workload, run the float64 oracle on the same inputs, and compare
with the tolerances fixed before looking at results:

* masks, lengths and advantages for binary rewards: bit-exact;
* scalar loss: within 1e-5 relative, with |delta| <= 1e-5 * max(|loss|, L1)
  where L1 = sum |ell_t| / norm (a loss that cancels to ~0 is judged against
  the size of its terms); exactly 0 when every term is 0;
* per-token log-probs: 2e-3 absolute for bfloat16 logits, 1e-5 for float32;
* dlogits: 1e-2 relative + 1e-6 absolute, skipping tokens whose oracle ratio
  lies within 1e-5 of a clip boundary (min() may take either branch there).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from vocab_wide_logprob_gb300 import workloads as wl

LOSS_RTOL = 1e-5
LOGP_ATOL = {"bf16": 2e-3, "f32": 1e-5}
DL_RTOL, DL_ATOL = 1e-2, 1e-6
KINK = 1e-5


def g():
    from vocab_wide_logprob_gb300 import _native
    return _native


def with_contrast(w: wl.Workload) -> wl.Workload:
    """The first of seeds seed, seed+1, ... whose rewards have contrast in at
    least one group (deterministic)."""
    k = 0
    while True:
        v = wl.variant(w, seed=w.seed + k)
        R = wl.make_rewards(v).reshape(v.B, v.G)
        if np.any(R.max(1) != R.min(1)):
            return v
        k += 1


def host_inputs(w: wl.Workload, lp_o: np.ndarray, m_o: np.ndarray):
    """old/ref log-probs = oracle log-probs + the generator's noise, as float32,
    NaN where the mask is 0 (those positions must never be read)."""
    n_old, n_ref = wl.make_noise(w)
    old = ref = None
    if n_old is not None:
        old = (lp_o + n_old).astype(np.float32)
        old[m_o == 0] = np.nan
    if n_ref is not None:
        ref = (lp_o + n_ref).astype(np.float32)
        ref[m_o == 0] = np.nan
    return old, ref


def dev(x, device="cuda"):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device)


def run_gpu(w: wl.Workload, logits, ids, R, old, ref, grad=None, dlogits=None, eps=None,
            beta=None, norm=0.0, fused=False, bwd_flags=0):
    """mask -> advantage -> fwd -> bwd (or the fused fwd+bwd) through the C
    ABI; returns tensors.  bwd_flags: grpo_loss_bwd_ex flags of the two-pass
    backward (GRPO_BWD_SKIP_ZERO_WEIGHT = 1)."""
    n = g()
    t_ids = dev(ids)
    mask, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(dev(R), w.G)
    gt = None if grad is None else torch.tensor([grad], dtype=torch.float32, device="cuda")
    e = w.eps if eps is None else eps
    b = w.beta if beta is None else beta
    if fused:
        out = n.grpo_loss_fwd_bwd(logits, w.P, t_ids, lens, adv, dev(old), dev(ref), e, b, norm,
                                  gt, dlogits=dlogits)
        dl = out["dlogits"]
    else:
        out = n.grpo_loss_fwd(logits, w.P, t_ids, lens, adv, dev(old), dev(ref), e, b, norm)
        if bwd_flags:
            dl = n.grpo_loss_bwd_ex(logits, w.P, t_ids, lens, out["lse"], out["w"], gt, dlogits,
                                    flags=bwd_flags)
        else:
            dl = n.grpo_loss_bwd(logits, w.P, t_ids, lens, out["lse"], out["w"], gt, dlogits)
    status = n.grpo_check_error(out["workspace"])
    torch.cuda.synchronize()
    out.update(mask=mask, lens=lens, adv=adv, dlogits=dl, status=status)
    return out


def kink_tokens(lp_o, old, eps):
    """Boolean [N, C]: oracle ratio within KINK of 1-eps or 1+eps."""
    if old is None:
        return np.zeros(lp_o.shape, bool)
    with np.errstate(invalid="ignore"):
        r = np.exp(lp_o - old.astype(np.float64))
        return (np.abs(r - (1 - eps)) < KINK) | (np.abs(r - (1 + eps)) < KINK)


def w_scale(lp_o, old, ref, A, beta, norm):
    """Size of the two terms of w (|A| r and beta exp(ref - logp)), per token:
    w's error is relative to this, since the terms can cancel."""
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.ones_like(lp_o) if old is None else np.exp(lp_o - old.astype(np.float64))
        e = np.zeros_like(lp_o) if ref is None else np.exp(ref.astype(np.float64) - lp_o)
        s = (np.abs(A)[:, None] * r + beta * (1.0 + e)) / norm
    return np.nan_to_num(s, nan=1.0)


def assert_loss(loss_gpu, loss_o, ell_o, norm):
    l1 = float(np.sum(np.abs(ell_o))) / norm
    if l1 == 0.0:
        assert loss_gpu == 0.0, (loss_gpu, loss_o)
        return
    tol = LOSS_RTOL * max(abs(loss_o), l1)
    assert abs(loss_gpu - loss_o) <= tol, (loss_gpu, loss_o, tol)


def assert_dlogits(d_gpu: np.ndarray, d_o: np.ndarray, where=""):
    d_gpu = d_gpu.astype(np.float64)
    err = np.abs(d_gpu - d_o)
    bad = err > DL_RTOL * np.abs(d_o) + DL_ATOL
    assert not np.any(bad), (where, int(bad.sum()), float(err.max()),
                             np.argwhere(bad)[:5].tolist())


def to_host_logits(t: torch.Tensor):
    return wl.logits_as_numpy(t.cpu())


def check_small(w: wl.Workload, logits_cpu=None, grad=None, norm=0.0, logits_gpu=None,
                fused=False, dlogits=None, bwd_flags=0):
    """Whole-batch element-wise comparison (sizes the oracle finishes fast)."""
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    if logits_cpu is None:
        logits_cpu = wl.make_logits_cpu(w)
    z, dt = wl.logits_as_numpy(logits_cpu)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage(R, w.G)
    lp_o, lse_o = oracle.logp(z, dt, w.P, w.C, ids, len_o)
    old, ref = host_inputs(w, lp_o, m_o)
    nrm = norm if norm > 0 else float(w.N * w.C)
    loss_o, w_o, ell_o = oracle.loss(lp_o, None if old is None else old.astype(np.float64),
                                     None if ref is None else ref.astype(np.float64), A_o,
                                     len_o, w.eps, w.beta, nrm)
    gval = 1.0 if grad is None else grad
    d_o = oracle.dlogits(z, dt, w.P, w.C, ids, len_o, lse_o, w_o, gval)

    logits = logits_cpu.cuda() if logits_gpu is None else logits_gpu
    out = run_gpu(w, logits, ids, R, old, ref, grad=grad, norm=norm, fused=fused,
                  dlogits=dlogits, bwd_flags=bwd_flags)
    assert out["status"] == 0
    assert np.array_equal(out["mask"].cpu().numpy(), m_o)
    assert np.array_equal(out["lens"].cpu().numpy(), len_o)
    adv = out["adv"].cpu().numpy()
    assert np.array_equal(adv, A_o.astype(np.float32)), (adv, A_o)
    lp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lp - lp_o)) <= LOGP_ATOL[dt], np.max(np.abs(lp - lp_o))
    lse = out["lse"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse - lse_o)) <= LOGP_ATOL[dt]
    assert np.all(lp[m_o == 0] == 0) and np.all(lse[m_o == 0] == 0)
    assert_loss(float(out["loss"].item()), loss_o, ell_o, nrm)
    kink = kink_tokens(lp_o, old, w.eps)
    wt = out["w"].cpu().numpy().astype(np.float64)
    ok = ~kink & (m_o == 1)
    scale = w_scale(lp_o, old, ref, A_o, w.beta, nrm)
    err = np.abs(wt - w_o)
    assert np.all(err[ok] <= 1e-4 * scale[ok] + 1e-12), (float(np.max(err[ok] / scale[ok])))
    d = out["dlogits"].float().cpu().numpy()
    rows_ok = np.ones((w.N, w.T), bool)
    for i, t in zip(*np.nonzero(kink)):
        rows_ok[i, w.P - 1 + t] = False
    assert_dlogits(d[rows_ok], d_o[rows_ok], w.name)
    return out, dict(loss=loss_o, w=w_o, lp=lp_o, lse=lse_o, len=len_o, A=A_o, kink=int(kink.sum()))


def oracle_logp_device_rows(w: wl.Workload, logits: torch.Tensor, ids, len_o):
    """Oracle log-probs over every valid row, copying one completion's scored
    rows to the host at a time (bounded host memory)."""
    lp_o = np.zeros((w.N, w.C))
    lse_o = np.zeros((w.N, w.C))
    for i in range(w.N):
        L = int(len_o[i])
        if L == 0:
            continue
        rows, dt = to_host_logits(logits[i, w.P - 1:w.P - 1 + L])
        lp, ls = oracle.logp_rows(rows, dt, ids[i, w.P:w.P + L])
        lp_o[i, :L] = lp
        lse_o[i, :L] = ls
    return lp_o, lse_o


def oracle_dlogits_rows(z, dt, y, lse, wt, g=1.0):
    """The oracle's gradient of k independent scored rows z [k, V] with
    targets y [k], log-sum-exps lse [k] and weights wt [k]: the rows laid out
    as a batch of one sequence (prompt length 1, so row t scores token t) and
    passed to :func:`oracle.dlogits`, which runs them on all host cores."""
    k, V = z.shape
    zb = np.concatenate([z, np.zeros((1, V), z.dtype)])[None]
    ids_b = np.concatenate([[0], np.asarray(y, np.int64)])[None]
    d = oracle.dlogits(zb, dt, 1, k, ids_b, np.array([k], np.int32),
                       np.asarray(lse, np.float64)[None], np.asarray(wt, np.float64)[None], g)
    return d[0, :k]


def check_full_size(w: wl.Workload, rows="all", grad=None, seed=0):
    """A full-size workload in the benchmark's launch configuration: the whole
    loss, every log-prob, the gradient of scored rows computed by the oracle
    one completion at a time (``rows="all"``: every scored row; ``"ends"``:
    the first, middle and last scored row of every completion), and every
    row that scores nothing checked to be +0 bit for bit."""
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    logits = torch.empty((w.N, w.T, w.V), dtype=torch.bfloat16 if w.dtype == "bf16"
                         else torch.float32, device="cuda")
    wl.fill_logits_cuda(w, logits)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    A_o = oracle.advantage(R, w.G)
    lp_o, lse_o = oracle_logp_device_rows(w, logits, ids, len_o)
    old, ref = host_inputs(w, lp_o, m_o)
    nrm = float(w.N * w.C)
    loss_o, w_o, ell_o = oracle.loss(lp_o, None if old is None else old.astype(np.float64),
                                     None if ref is None else ref.astype(np.float64), A_o,
                                     len_o, w.eps, w.beta, nrm)
    out = run_gpu(w, logits, ids, R, old, ref, grad=grad)
    gval = 1.0 if grad is None else grad
    assert out["status"] == 0
    assert np.array_equal(out["mask"].cpu().numpy(), m_o)
    assert np.array_equal(out["lens"].cpu().numpy(), len_o)
    assert np.array_equal(out["adv"].cpu().numpy(), A_o.astype(np.float32))
    lp = out["logp"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lp - lp_o)) <= LOGP_ATOL[w.dtype], np.max(np.abs(lp - lp_o))
    lse_gpu = out["lse"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse_gpu - lse_o)) <= LOGP_ATOL[w.dtype]
    assert_loss(float(out["loss"].item()), loss_o, ell_o, nrm)
    kink = kink_tokens(lp_o, old, w.eps)

    dl = out["dlogits"]
    compared = 0
    for i in range(w.N):
        L = int(len_o[i])
        if L == 0:
            continue
        ts = np.arange(L) if rows == "all" else np.unique([0, L // 2, L - 1])
        ts = ts[~kink[i, ts]]
        if len(ts) == 0:
            continue
        sel = torch.from_numpy(w.P - 1 + ts).to(logits.device)
        z, dt = to_host_logits(logits[i].index_select(0, sel))
        y = ids[i, w.P + ts]
        d_o = oracle_dlogits_rows(z, dt, y, lse_o[i, ts], w_o[i, ts], gval)
        d_g, _ = to_host_logits(dl[i].index_select(0, sel))
        assert_dlogits(_as_f64(d_g, dt), d_o, f"{w.name} completion {i}")
        compared += len(ts)
    # rows that score nothing: prompt rows 0..P-2, rows past each length,
    # the last row; +0 exactly (bit pattern 0)
    bits = dl.view(torch.int16 if dl.dtype == torch.bfloat16 else torch.int32)
    zero_rows = 0
    for i in range(w.N):
        first = w.P - 1 + int(len_o[i])
        assert not bool(bits[i, :w.P - 1].any()), (w.name, i, "prompt rows")
        assert not bool(bits[i, first:].any()), (w.name, i, "rows past the length")
        zero_rows += (w.P - 1) + (w.T - first)
    torch.cuda.synchronize()
    return out, dict(loss=loss_o, compared=compared, zero_rows=zero_rows,
                     kink=int(kink.sum()), logits=logits, ids=ids, w_o=w_o, lse_o=lse_o,
                     len_o=len_o)


def _as_f64(a, dt):
    if dt == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
