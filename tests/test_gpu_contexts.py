"""The library in a second CUDA context on the same device.

The static scratch's device address and the per-stream call record are kept
per CUDA context, and the kernels' raised shared-memory limits are set per
context.  A child process runs the calls first in the device's primary
context (through the Python binding), then in a second context it creates
with the driver API (through the C ABI, on that context's default stream,
with buffers from cuMemAlloc), and the two runs must give the same bits:
the log-sum-exp, single-pass, static-scratch, LM-head log-prob and LM-head
loss forward and backward kernels, each of which needs more than the default
48 KiB of shared memory."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_second_context_same_bits():
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--child"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    assert "second context: same bits" in r.stdout


def _child():
    import torch

    sys.path.insert(0, ROOT)
    from vocab_wide_logprob_gb300 import _native as g

    N, P, C, V, d = 4, 8, 64, 32000, 128
    T = P + C
    rng = np.random.default_rng(7)
    logits = torch.from_numpy(rng.normal(0, 3, (N, T, V)).astype(np.float32)).to(torch.bfloat16)
    ids = rng.integers(0, V, (N, T), dtype=np.int64)
    lens = np.array([C, 17, 1, 40], dtype=np.int32)
    adv = np.array([0.5, -0.5, 0.25, -0.25], dtype=np.float32)
    old = rng.normal(-10, 1, (N, C)).astype(np.float32)
    hidden = torch.from_numpy(rng.normal(0, 1, (N, T, d)).astype(np.float32)).to(torch.bfloat16)
    weight = torch.from_numpy(rng.normal(0, 0.05, (V, d)).astype(np.float32)).to(torch.bfloat16)
    eps, beta, norm = 0.2, 0.0, 0.0

    # ---- primary context, through the binding ---------------------------------
    dev = torch.device("cuda")
    t_logits, t_hidden, t_weight = logits.to(dev), hidden.to(dev), weight.to(dev)
    t_ids, t_lens = torch.from_numpy(ids).to(dev), torch.from_numpy(lens).to(dev)
    t_adv, t_old = torch.from_numpy(adv).to(dev), torch.from_numpy(old).to(dev)
    ref = {}
    lp, lse, _ = g.grpo_logprobs(t_logits, P, t_ids, t_lens)
    ref["logprobs"] = (lp.cpu().numpy(), lse.cpu().numpy())
    out = g.grpo_loss_fwd_bwd(t_logits, P, t_ids, t_lens, t_adv, t_old, None, eps, beta, norm)
    ref["fused"] = (out["logp"].cpu().numpy(), out["w"].cpu().numpy(),
                    out["loss"].cpu().numpy(), out["dlogits"].view(torch.int16).cpu().numpy())
    st = g.grpo_loss_fwd_static(t_logits, P, t_ids, t_lens, t_adv, t_old, None, eps, beta, norm)
    ref["static"] = (st["logp"].cpu().numpy(), st["loss"].cpu().numpy())
    lp2, lse2, _ = g.grpo_lmhead_logprobs(t_hidden, t_weight, P, t_ids, t_lens)
    ref["lmhead_logprobs"] = (lp2.cpu().numpy(),)
    f = g.grpo_lmhead_loss_fwd(t_hidden, t_weight, P, t_ids, t_lens, t_adv, t_old, None, eps,
                               beta, norm)
    dh, dw, _ = g.grpo_lmhead_loss_bwd(t_hidden, t_weight, P, t_ids, t_lens, f["lse"], f["w"])
    ref["lmhead_loss"] = (f["w"].cpu().numpy(), f["loss"].cpu().numpy(), dh.cpu().numpy(),
                          dw.cpu().numpy())
    torch.cuda.synchronize()

    # ---- a second context on the same device, through the C ABI --------------
    lib = g.library()
    cu = ctypes.CDLL("libcuda.so.1")

    def ck(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: CUresult {rc}")

    ck(cu.cuInit(0), "cuInit")
    cudev = ctypes.c_int()
    ck(cu.cuCtxGetDevice(ctypes.byref(cudev)), "cuCtxGetDevice")
    ctx = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), ctypes.c_uint(0), cudev), "cuCtxCreate")  # current
    bufs = []

    def alloc(nbytes):
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(int(nbytes), 16))), "cuMemAlloc")
        bufs.append(p.value)
        return ctypes.c_void_p(p.value)

    def put(arr):
        arr = np.ascontiguousarray(arr)
        p = alloc(arr.nbytes)
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p.value), arr.ctypes.data_as(ctypes.c_void_p),
                              ctypes.c_size_t(arr.nbytes)), "cuMemcpyHtoD")
        return p

    def get(p, shape, dtype):
        arr = np.empty(shape, dtype=dtype)
        ck(cu.cuMemcpyDtoH_v2(arr.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(p.value),
                              ctypes.c_size_t(arr.nbytes)), "cuMemcpyDtoH")
        return arr

    def ok(status, what):
        if status != 0:
            raise RuntimeError(f"{what} in the second context: status {status}")

    def size(fn, *args):
        out = ctypes.c_size_t()
        ok(fn(*args, ctypes.byref(out)), fn.__name__)
        return out.value

    s0 = None  # the current context's default stream
    d_logits = put(logits.view(torch.int16).numpy())
    d_hidden = put(hidden.view(torch.int16).numpy())
    d_weight = put(weight.view(torch.int16).numpy())
    d_ids, d_lens, d_adv, d_old = put(ids), put(lens), put(adv), put(old)
    ws_bytes = size(lib.grpo_workspace_size, N, C, V)
    nc = (N, C)

    lp_, lse_, ws = alloc(4 * N * C), alloc(4 * N * C), alloc(ws_bytes)
    ok(lib.grpo_logprobs(d_logits, g.GRPO_BF16, N, P, C, V, d_ids, d_lens, lp_, lse_, ws,
                         ws_bytes, s0), "grpo_logprobs")

    f_lp, f_lse, f_w, f_loss = alloc(4 * N * C), alloc(4 * N * C), alloc(4 * N * C), alloc(4)
    f_dl, ws2 = alloc(2 * N * T * V), alloc(ws_bytes)
    ok(lib.grpo_loss_fwd_bwd(d_logits, g.GRPO_BF16, N, P, C, V, d_ids, d_lens, d_adv, d_old,
                             None, eps, beta, norm, None, f_lp, f_lse, f_w, f_loss, f_dl, ws2,
                             ws_bytes, s0), "grpo_loss_fwd_bwd")

    s_lp, s_lse, s_w, s_loss = alloc(4 * N * C), alloc(4 * N * C), alloc(4 * N * C), alloc(4)
    ok(lib.grpo_loss_fwd_static(d_logits, g.GRPO_BF16, N, P, C, V, d_ids, d_lens, d_adv, d_old,
                                None, eps, beta, norm, s_lp, s_lse, s_w, s_loss, s0),
       "grpo_loss_fwd_static")

    lws_bytes = size(lib.grpo_lmhead_workspace_size, N, C, V, d)
    m_lp, m_lse, lws = alloc(4 * N * C), alloc(4 * N * C), alloc(lws_bytes)
    ok(lib.grpo_lmhead_logprobs(d_hidden, d_weight, N, P, C, V, d, d_ids, d_lens, m_lp, m_lse,
                                lws, lws_bytes, s0), "grpo_lmhead_logprobs")

    l_lp, l_lse, l_w, l_loss = alloc(4 * N * C), alloc(4 * N * C), alloc(4 * N * C), alloc(4)
    lws2 = alloc(lws_bytes)
    ok(lib.grpo_lmhead_loss_fwd(d_hidden, d_weight, N, P, C, V, d, d_ids, d_lens, d_adv, d_old,
                                None, eps, beta, norm, l_lp, l_lse, l_w, l_loss, lws2, lws_bytes,
                                s0), "grpo_lmhead_loss_fwd")
    bws_bytes = size(lib.grpo_lmhead_bwd_workspace_size, N, C, V, d)
    l_dh, l_dw, bws = alloc(4 * N * T * d), alloc(4 * V * d), alloc(bws_bytes)
    ok(lib.grpo_lmhead_loss_bwd(d_hidden, d_weight, N, P, C, V, d, d_ids, d_lens, l_lse, l_w,
                                None, l_dh, l_dw, bws, bws_bytes, s0), "grpo_lmhead_loss_bwd")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    for w_ in (ws, ws2, lws, lws2, bws):
        ok(lib.grpo_check_error(w_, s0), "grpo_check_error")

    cmp = {
        "logprobs": ((get(lp_, nc, np.float32), get(lse_, nc, np.float32)), ref["logprobs"]),
        "fused": ((get(f_lp, nc, np.float32), get(f_w, nc, np.float32),
                   get(f_loss, (1,), np.float32), get(f_dl, (N, T, V), np.int16)), ref["fused"]),
        "static": ((get(s_lp, nc, np.float32), get(s_loss, (1,), np.float32)), ref["static"]),
        "lmhead_logprobs": ((get(m_lp, nc, np.float32),), ref["lmhead_logprobs"]),
        "lmhead_loss": ((get(l_w, nc, np.float32), get(l_loss, (1,), np.float32),
                         get(l_dh, (N, T, d), np.float32), get(l_dw, (V, d), np.float32)),
                        ref["lmhead_loss"]),
    }
    for p in bufs:
        cu.cuMemFree_v2(ctypes.c_uint64(p))
    popped = ctypes.c_void_p()
    ck(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
    ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
    for name, (a, b) in cmp.items():
        for k, (x, y) in enumerate(zip(a, b)):
            xv = x.view(np.uint32) if x.dtype == np.float32 else x
            yv = y.view(np.uint32) if y.dtype == np.float32 else y
            if not np.array_equal(xv, yv):
                raise AssertionError(f"{name}[{k}] differs between the two contexts")
    print("second context: same bits")


if __name__ == "__main__" and "--child" in sys.argv:
    _child()
