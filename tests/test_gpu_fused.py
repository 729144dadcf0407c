"""The fused forward+backward (grpo_loss_fwd_bwd) against the float64 oracle
and against the two-call path: logp, lse, w and dlogits must have the same
bits as grpo_loss_fwd followed by grpo_loss_bwd (same arithmetic per element,
same per-token terms); the loss is summed in another fixed order and must
agree to float rounding."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _both(w, logits_cpu=None, grad=None, norm=0.0, logits_gpu=None, dlogits=None):
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    if logits_cpu is None:
        logits_cpu = wl.make_logits_cpu(w)
    z, dt = wl.logits_as_numpy(logits_cpu)
    m_o, len_o = oracle.mask(ids, w.P, w.C, w.eos_id)
    lp_o, _ = oracle.logp(z, dt, w.P, w.C, ids, len_o)
    old, ref = H.host_inputs(w, lp_o, m_o)
    logits = logits_cpu.cuda() if logits_gpu is None else logits_gpu
    a = H.run_gpu(w, logits, ids, R, old, ref, grad=grad, norm=norm)
    b = H.run_gpu(w, logits, ids, R, old, ref, grad=grad, norm=norm, fused=True, dlogits=dlogits)
    return a, b


CASES = [
    wl.variant(wl.TINY, name="tiny_terms", old_sigma=0.1, ref_sigma=0.1, beta=0.04),
    wl.variant(wl.QWEN_G8, name="bf16_small", B=1, G=4, P=8, C=24, reward_p=0.5,
               old_sigma=0.1, ref_sigma=0.1, beta=0.04, trunc=0.25, seed=77),
    wl.variant(wl.TINY, name="ragged_bf16", V=50001, dtype="bf16", old_sigma=0.1,
               ref_sigma=0.1, beta=0.04, logit_std=3.0, seed=11),
    wl.variant(wl.TINY, name="ragged_f32", V=65539, dtype="f32", old_sigma=0.1, ref_sigma=0.1,
               beta=0.04, logit_std=3.0, seed=12),
    wl.variant(wl.TINY, name="tiny_V7", V=7, dtype="bf16", old_sigma=0.1, seed=13),
    wl.variant(wl.TINY, name="C1", C=1, old_sigma=0.1, ref_sigma=0.1, beta=0.04),
    wl.variant(wl.TINY, name="G32", G=32, B=2, reward_p=0.5, old_sigma=0.1),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_matches_oracle(w):
    H.check_small(H.with_contrast(w), fused=True)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_same_bits_as_two_calls(w):
    a, b = _both(H.with_contrast(w), grad=3.0)
    for k in ("logp", "lse", "w", "dlogits", "mask", "lens", "adv"):
        x, y = a[k], b[k]
        if x.dtype in (torch.float32, torch.bfloat16):
            assert torch.equal(_bits(x), _bits(y)), k
        else:
            assert torch.equal(x, y), k
    la, lb = float(a["loss"].item()), float(b["loss"].item())
    assert abs(la - lb) <= 1e-6 * max(abs(la), 1e-12), (la, lb)


@pytest.mark.parametrize("B,C,V,dtype", [(50, 4, 50001, "bf16"), (1025, 1, 50000, "bf16"),
                                         (50, 4, 20001, "f32")],
                         ids=["N200_two_head_slots", "N4100_offsets_in_memory", "N200_f32"])
def test_fused_head_slots_same_bits(B, C, V, dtype):
    """The fused kernel holds each row's first chunks in shared-memory slots,
    as many as fit beside its ring and offsets table with two CTAs per SM:
    two at 200 completions, three again at 4,100 (the offsets table then
    stays in global memory).  Whole rows per CTA (N*C above four rows per
    SM), five to seven 16 KiB chunks a row, so the ring carries the rest;
    the outputs have the bits of the two calls."""
    w = H.with_contrast(wl.variant(wl.TINY, name=f"slots_N{4 * B}_{dtype}", B=B, G=4, P=1, C=C,
                                   V=V, dtype=dtype, logit_std=3.0, seed=500 + B))
    logits = torch.empty((w.N, w.T, w.V), device="cuda",
                         dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    wl.fill_logits_cuda(w, logits)
    ids, R = wl.make_ids(w), wl.make_rewards(w)
    a = H.run_gpu(w, logits, ids, R, None, None, grad=1.5, beta=0.0)
    b = H.run_gpu(w, logits, ids, R, None, None, grad=1.5, beta=0.0, fused=True)
    assert a["status"] == 0 and b["status"] == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert w.N * w.C >= 4 * sms and int(a["lens"].sum()) >= 2 * sms
    for k in ("logp", "lse", "w", "dlogits"):
        assert torch.equal(_bits(a[k]), _bits(b[k])), k
    la, lb = float(a["loss"].item()), float(b["loss"].item())
    assert abs(la - lb) <= 1e-6 * max(abs(la), 1e-12), (la, lb)


def test_fused_scaled_gradient():
    w = wl.variant(wl.TINY, old_sigma=0.1, ref_sigma=0.1, beta=0.04)
    H.check_small(w, grad=float(w.N * w.C), fused=True)


def test_fused_phase_mismatch_falls_back():
    """dlogits one element off the logits' 16-byte phase: the call runs the
    two passes; results still match the oracle."""
    w = wl.variant(wl.TINY, name="phase", V=1000, dtype="bf16", old_sigma=0.1, seed=99)
    base = torch.empty(w.N * w.T * w.V + 1, dtype=torch.bfloat16, device="cuda")
    H.check_small(w, fused=True, dlogits=base[1:].view(w.N, w.T, w.V))


def test_fused_reports_bad_token():
    w = wl.TINY
    ids = wl.make_ids(w)
    ids[0, w.P + 3] = -1
    g = H.g()
    logits = wl.make_logits_cpu(w).cuda()
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = torch.zeros((w.N,), device="cuda")
    out = g.grpo_loss_fwd_bwd(logits, w.P, t_ids, lens, adv)
    assert g.grpo_check_error(out["workspace"]) == 6
    assert np.isnan(out["logp"].cpu().numpy()[0, 3])


@pytest.mark.parametrize("w", [wl.QWEN_G8, wl.BATCHED], ids=lambda w: w.name)
def test_fused_full_size_same_bits(w):
    w = H.with_contrast(w)
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    logits = torch.empty((w.N, w.T, w.V), dtype=torch.bfloat16, device="cuda")
    wl.fill_logits_cuda(w, logits)
    n_old, n_ref = wl.make_noise(w)
    g = H.g()
    t_ids = torch.from_numpy(ids).cuda()
    _, lens = g.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = g.grpo_advantage(torch.from_numpy(R).cuda(), w.G)
    cur = g.grpo_loss_fwd(logits, w.P, t_ids, lens, adv)
    old = cur["logp"] + torch.from_numpy(n_old).float().cuda()
    a = g.grpo_loss_fwd(logits, w.P, t_ids, lens, adv, old, None, w.eps, w.beta)
    da = g.grpo_loss_bwd(logits, w.P, t_ids, lens, a["lse"], a["w"])
    b = g.grpo_loss_fwd_bwd(logits, w.P, t_ids, lens, adv, old, None, w.eps, w.beta)
    torch.cuda.synchronize()
    assert g.grpo_check_error(b["workspace"]) == 0
    for k in ("logp", "lse", "w"):
        assert torch.equal(_bits(a[k]), _bits(b[k])), k
    assert torch.equal(_bits(da), _bits(b["dlogits"]))
    la, lb = float(a["loss"].item()), float(b["loss"].item())
    assert abs(la - lb) <= 1e-6 * max(abs(la), 1e-12), (la, lb)
    del logits, da, b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("host_dl", [False, True], ids=["dev_dlogits", "host_dlogits"])
@pytest.mark.parametrize("dtype,V,shift", [("bf16", 1024, 0), ("bf16", 1001, 0), ("f32", 1001, 0),
                                           ("bf16", 1024, 1), ("f32", 1001, 1)],
                         ids=["bf16_vec16", "bf16_odd_V", "f32_odd_V", "bf16_host_phase_shift",
                              "f32_host_phase_shift"])
def test_host_logits_match_device_path(dtype, V, shift, host_dl):
    """grpo_loss_fwd_bwd_host on pinned host logits gives the bits of
    grpo_loss_fwd_bwd on the same logits in device memory, and only the
    scored rows of the staging buffer are written.  With the host buffer in
    the staging buffer's 16-byte phase the gradient kernel reads the host rows
    itself (ragged heads and tails for odd V); shifted by `shift` elements, the
    rows are gathered first (16-byte, 4-byte and 2-byte copy units)."""
    n = H.g()
    w = H.with_contrast(wl.variant(wl.QWEN_G8, name=f"host_{dtype}_{V}", B=2, G=4, P=6, C=20,
                                   V=V, eos_id=V - 1, dtype=dtype, seed=91))
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    logits = wl.make_logits_cpu(w)
    t_ids = H.dev(ids)
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(R), w.G)
    rng = np.random.default_rng(4)
    old = torch.from_numpy(rng.normal(-7, 1, (w.N, w.C)).astype(np.float32)).cuda()
    a = n.grpo_loss_fwd_bwd(logits.cuda(), w.P, t_ids, lens, adv, old, None, 0.2, 0.0)
    staging = torch.full(logits.shape, 7.0, dtype=logits.dtype, device="cuda")
    host = logits.pin_memory()
    if shift:
        buf = torch.empty(logits.numel() + shift, dtype=logits.dtype).pin_memory()
        host = buf[shift:].view(logits.shape)
        host.copy_(logits)
        assert host.is_pinned() and host.data_ptr() % 16 != 0
    dl_out = None
    if host_dl:  # the gradient written straight into pinned host memory
        dl_out = torch.full(logits.shape, 5.0, dtype=logits.dtype).pin_memory()
    b = n.grpo_loss_fwd_bwd_host(host, w.P, t_ids, lens, adv, old, None, 0.2, 0.0,
                                 staging=staging, dlogits=dl_out)
    assert n.grpo_check_error(b["workspace"]) == 0
    assert b["dlogits"].is_cuda != host_dl
    for k in ("logp", "lse", "w", "loss"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["dlogits"].view(torch.int16 if dtype == "bf16" else torch.int32).cpu(),
                       b["dlogits"].view(torch.int16 if dtype == "bf16" else torch.int32).cpu())
    L = lens.cpu().numpy()
    scored = np.zeros((w.N, w.T), bool)
    for i in range(w.N):
        scored[i, w.P - 1:w.P - 1 + L[i]] = True
    st = staging.float().cpu().numpy()
    assert np.array_equal(st[scored], logits.float().numpy()[scored])
    assert np.all(st[~scored] == 7.0)


def test_host_logits_refuses_pageable_memory():
    """Pageable host memory is not addressable by the device: refused before
    any launch."""
    import ctypes
    n = H.g()
    lib = n.library()
    buf = np.zeros((2, 8, 64), np.float32)
    dev = torch.zeros((64,), dtype=torch.uint8, device="cuda")
    dl = torch.zeros((2, 8, 64), dtype=torch.float32, device="cuda")
    st = torch.zeros((2, 8, 64), dtype=torch.float32, device="cuda")
    ws = torch.zeros((1 << 16,), dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p
    rc = lib.grpo_loss_fwd_bwd_host(p(buf.ctypes.data), 0, 2, 4, 4, 64, p(dev.data_ptr()),
                                    p(dev.data_ptr()), p(dev.data_ptr()), None, None, 0.2, 0.0, 0.0,
                                    None, p(dev.data_ptr()), p(dev.data_ptr()),
                                    p(dev.data_ptr()), p(dev.data_ptr()), p(dl.data_ptr()),
                                    p(st.data_ptr()), p(ws.data_ptr()), ws.numel(), None)
    assert rc == 1  # GRPO_ERR_INVALID_ARG


def test_host_logits_registered_too_short():
    """A host buffer page-locked over only part of the logits' size is refused
    before anything is enqueued (the kernels read any scored row, up to the
    last byte); the same buffer page-locked in full is accepted and gives the
    bits of the device-memory path."""
    import ctypes
    n = H.g()
    lib = n.library()
    w = H.with_contrast(wl.variant(wl.QWEN_G8, name="short_host", B=2, G=4, P=6, C=26, V=1024,
                                   eos_id=1023, seed=92))
    logits = wl.make_logits_cpu(w)
    nbytes = logits.numel() * 2
    assert nbytes % 8192 == 0
    raw = np.zeros(nbytes + 4096, np.uint8)
    off = (-raw.ctypes.data) % 4096
    buf = raw[off:off + nbytes]
    buf[:] = logits.view(torch.int16).numpy().view(np.uint8).reshape(-1)
    t_ids = H.dev(wl.make_ids(w))
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(wl.make_rewards(w)), w.G)
    ref = n.grpo_loss_fwd_bwd(logits.cuda(), w.P, t_ids, lens, adv, None, None, 0.2, 0.0)
    out = {k: torch.empty_like(ref[k]) for k in ("logp", "lse", "w", "loss")}
    dl = torch.empty((w.N, w.T, w.V), dtype=torch.bfloat16, device="cuda")
    st = torch.empty_like(dl)
    ws = torch.zeros((n.grpo_workspace_size(w.N, w.C, w.V),), dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return lib.grpo_loss_fwd_bwd_host(
            p(buf.ctypes.data), 1, w.N, w.P, w.C, w.V, p(t_ids.data_ptr()), p(lens.data_ptr()),
            p(adv.data_ptr()), None, None, 0.2, 0.0, 0.0, None, p(out["logp"].data_ptr()),
            p(out["lse"].data_ptr()), p(out["w"].data_ptr()), p(out["loss"].data_ptr()),
            p(dl.data_ptr()), p(st.data_ptr()), p(ws.data_ptr()), ws.numel(), p(stream))

    cudart = torch.cuda.cudart()
    flags = 3  # cudaHostRegisterPortable | cudaHostRegisterMapped
    for registered in (nbytes // 2, nbytes - 4096):
        assert int(cudart.cudaHostRegister(buf.ctypes.data, registered, flags)) == 0
        try:
            assert call() == 1  # GRPO_ERR_INVALID_ARG, nothing enqueued
        finally:
            assert int(cudart.cudaHostUnregister(buf.ctypes.data)) == 0
    assert int(cudart.cudaHostRegister(buf.ctypes.data, nbytes, flags)) == 0
    try:
        assert call() == 0
        torch.cuda.synchronize()
    finally:
        assert int(cudart.cudaHostUnregister(buf.ctypes.data)) == 0
    assert n.grpo_check_error(ws) == 0
    for k in ("logp", "lse", "w", "loss"):
        assert torch.equal(_bits(ref[k]), _bits(out[k])), k
    assert torch.equal(_bits(ref["dlogits"]), _bits(dl))


def test_host_dlogits_refused_when_short_or_pageable():
    """A host dlogits buffer must be page-locked over the whole gradient:
    pageable memory, a buffer page-locked over only its first part, and one
    overlapping the host logits are refused before anything is enqueued."""
    n = H.g()
    w = H.with_contrast(wl.variant(wl.QWEN_G8, name="short_dl", B=2, G=4, P=6, C=26, V=1024,
                                   eos_id=1023, seed=93))
    host = wl.make_logits_cpu(w).pin_memory()
    t_ids = H.dev(wl.make_ids(w))
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(H.dev(wl.make_rewards(w)), w.G)
    nbytes = host.numel() * 2
    raw = np.zeros(nbytes + 4096, np.uint8)
    off = (-raw.ctypes.data) % 4096
    buf = raw[off:off + nbytes]
    dl_view = torch.from_numpy(buf).view(torch.bfloat16).view(host.shape)
    # pageable: the binding refuses it, and so does the library
    with pytest.raises(ValueError):
        n.grpo_loss_fwd_bwd_host(host, w.P, t_ids, lens, adv, dlogits=dl_view)
    import ctypes
    lib = n.library()
    ws = torch.zeros((n.grpo_workspace_size(w.N, w.C, w.V),), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((w.N, w.C), device="cuda") for _ in range(3)] + \
        [torch.empty((1,), device="cuda")]
    st = torch.empty(host.shape, dtype=host.dtype, device="cuda")
    p = ctypes.c_void_p
    stream = torch.cuda.current_stream().cuda_stream

    def call(dl_ptr):
        return lib.grpo_loss_fwd_bwd_host(
            p(host.data_ptr()), 1, w.N, w.P, w.C, w.V, p(t_ids.data_ptr()), p(lens.data_ptr()),
            p(adv.data_ptr()), None, None, 0.2, 0.0, 0.0, None, *[p(t.data_ptr()) for t in outs],
            p(dl_ptr), p(st.data_ptr()), p(ws.data_ptr()), ws.numel(), p(stream))

    assert call(buf.ctypes.data) == 1
    cudart = torch.cuda.cudart()
    assert int(cudart.cudaHostRegister(buf.ctypes.data, nbytes // 2, 3)) == 0
    try:
        assert call(buf.ctypes.data) == 1   # page-locked over half its size only
    finally:
        assert int(cudart.cudaHostUnregister(buf.ctypes.data)) == 0
    assert call(host.data_ptr() + 4096) == 1  # overlaps the host logits
    torch.cuda.synchronize()


def test_host_logits_full_size_same_bits():
    """The benchmark workload (V = 151,936, whole rows per CTA) with the logits
    in pinned host memory: the gradient kernel reads the scored rows from host
    memory itself, and every output has the bits of the device-memory path."""
    n = H.g()
    w = H.with_contrast(wl.QWEN_G8)
    logits = torch.empty((w.N, w.T, w.V), dtype=torch.bfloat16, device="cuda")
    wl.fill_logits_cuda(w, logits)
    t_ids = torch.from_numpy(wl.make_ids(w)).cuda()
    _, lens = n.grpo_mask(t_ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(torch.from_numpy(wl.make_rewards(w)).cuda(), w.G)
    a = n.grpo_loss_fwd_bwd(logits, w.P, t_ids, lens, adv, None, None, 0.2, 0.0)
    host = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    host.copy_(logits)
    staging = torch.empty_like(logits)
    b = n.grpo_loss_fwd_bwd_host(host, w.P, t_ids, lens, adv, None, None, 0.2, 0.0,
                                 staging=staging)
    torch.cuda.synchronize()
    assert n.grpo_check_error(b["workspace"]) == 0
    for k in ("logp", "lse", "w", "loss"):
        assert torch.equal(_bits(a[k]), _bits(b[k])), k
    assert torch.equal(_bits(a["dlogits"]), _bits(b["dlogits"]))
    # the gradient written straight into pinned host memory: the same bits
    h_dl = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    c = n.grpo_loss_fwd_bwd_host(host, w.P, t_ids, lens, adv, None, None, 0.2, 0.0,
                                 staging=staging, dlogits=h_dl)
    torch.cuda.synchronize()
    assert n.grpo_check_error(c["workspace"]) == 0
    assert torch.equal(_bits(a["loss"]), _bits(c["loss"]))
    assert torch.equal(_bits(a["dlogits"]).cpu(), _bits(h_dl))
    del logits, staging, host, a, b, c, h_dl
    torch.cuda.empty_cache()
