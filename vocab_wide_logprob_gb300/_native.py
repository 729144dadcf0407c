"""ctypes binding of ``libgrpo.so`` (the C ABI declared in ``include/grpo.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these calls.  Functions take PyTorch tensors for device
memory, pass ``tensor.data_ptr()`` and the current CUDA stream, and raise
:class:`GrpoError` on any status other than ``GRPO_OK``.  There is no CPU
fallback: importing this module fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_PKG, "libgrpo.so")

GRPO_OK = 0
STATUS_NAMES = {
    0: "GRPO_OK", 1: "GRPO_ERR_INVALID_ARG", 2: "GRPO_ERR_UNSUPPORTED",
    3: "GRPO_ERR_WORKSPACE", 4: "GRPO_ERR_MISALIGNED", 5: "GRPO_ERR_CUDA",
    6: "GRPO_ERR_TOKEN_RANGE", 7: "GRPO_ERR_LENGTH_RANGE", 8: "GRPO_ERR_TIMEOUT",
}
GRPO_F32, GRPO_BF16 = 0, 1
GRPO_ADV_DR, GRPO_ADV_STD = 0, 1
GRPO_AGG_TOKEN_SUM, GRPO_AGG_SEQ_MEAN = 0, 1
GRPO_BWD_SKIP_ZERO_WEIGHT = 1


class GrpoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_lib.grpo_status_string(status).decode()})")


def _load():
    if not os.path.exists(LIBRARY):
        raise ImportError(
            f"{LIBRARY} is missing: build it with `python -m vocab_wide_logprob_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIBRARY)
    P, I64, F, SZ, INT = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t,
                          ctypes.c_int)
    sig = {
        "grpo_status_string": ([INT], ctypes.c_char_p),
        "grpo_mask": ([P, I64, I64, I64, I64, P, P, P], INT),
        "grpo_advantage": ([P, I64, I64, P, P], INT),
        "grpo_workspace_size": ([I64, I64, I64, ctypes.POINTER(SZ)], INT),
        "grpo_loss_fwd": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P, P, SZ,
                           P], INT),
        "grpo_loss_bwd": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, P, P], INT),
        "grpo_check_error": ([P, P], INT),
        "grpo_selftest_timeout": ([P, P], INT),
        "grpo_set_early_start": ([ctypes.c_int], None),
        "grpo_copy": ([P, P, SZ, P], INT),
        "grpo_loss_fwd_static": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P,
                                  P], INT),
        "grpo_loss_fwd_bwd": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P, P,
                               P, P, SZ, P], INT),
        "grpo_loss_fwd_bwd_host": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P,
                                    P, P, P, P, SZ, P], INT),
        "grpo_advantage_ex": ([P, I64, I64, INT, F, P, P, P], INT),
        "grpo_loss_fwd_ex": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, INT, P, P, P, P,
                              P, SZ, P], INT),
        "grpo_loss_fwd_bwd_ex": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, INT, P, P,
                                  P, P, P, P, P, SZ, P], INT),
        "grpo_loss_bwd_ex": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, P, ctypes.c_uint32, P],
                             INT),
        "grpo_logprobs": ([P, INT, I64, I64, I64, I64, P, P, P, P, P, SZ, P], INT),
        "grpo_lmhead_workspace_size": ([I64, I64, I64, I64, ctypes.POINTER(SZ)], INT),
        "grpo_lmhead_logprobs": ([P, P, I64, I64, I64, I64, I64, P, P, P, P, P, SZ, P], INT),
        "grpo_lmhead_loss_fwd": ([P, P, I64, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P,
                                  P, SZ, P], INT),
        "grpo_lmhead_loss_fwd_ex": ([P, P, I64, I64, I64, I64, I64, P, P, P, P, P, F, F, F, INT, P,
                                     P, P, P, P, SZ, P], INT),
        "grpo_lmhead_bwd_workspace_size": ([I64, I64, I64, I64, ctypes.POINTER(SZ)], INT),
        "grpo_lmhead_bwd_workspace_size_rows": ([I64, I64, I64, I64, I64, ctypes.POINTER(SZ)],
                                                INT),
        "grpo_lmhead_loss_bwd_ex": ([P, P, I64, I64, I64, I64, I64, P, P, P, P, P, P, P,
                                     ctypes.c_uint32, P, SZ, P], INT),
        "grpo_lmhead_loss_bwd": ([P, P, I64, I64, I64, I64, I64, P, P, P, P, P, P, P, P, SZ, P],
                                 INT),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, where: str):
    if status != GRPO_OK:
        raise GrpoError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GRPO_F32
    if t.dtype == torch.bfloat16:
        return GRPO_BF16
    raise TypeError(f"logits dtype {t.dtype} is not supported (float32 or bfloat16)")


def _dev(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def grpo_mask(input_ids: torch.Tensor, P: int, C: int, eos_id: int, mask=None, len_out=None,
              stream=None):
    """Completion mask of ``input_ids`` [N, P+C] int64 -> ``(mask u8 [N, C],
    len int32 [N])``."""
    _dev(input_ids, "input_ids", torch.int64)
    N = input_ids.shape[0]
    if mask is None:
        mask = torch.empty((N, C), dtype=torch.uint8, device=input_ids.device)
    if len_out is None:
        len_out = torch.empty((N,), dtype=torch.int32, device=input_ids.device)
    _check(_lib.grpo_mask(_ptr(input_ids), N, P, C, int(eos_id), _ptr(mask), _ptr(len_out),
                          _stream(stream)), "grpo_mask")
    return mask, len_out


def grpo_advantage(rewards: torch.Tensor, G: int, adv=None, stream=None):
    """Dr. GRPO advantage: R_i minus its group's mean, float32 [B*G]."""
    _dev(rewards, "rewards", torch.float32)
    if adv is None:
        adv = torch.empty_like(rewards)
    n = rewards.numel()
    if G < 1 or n % G:
        raise ValueError("len(rewards) must be a multiple of G >= 1")
    _check(_lib.grpo_advantage(_ptr(rewards), n // G, G, _ptr(adv), _stream(stream)),
           "grpo_advantage")
    return adv


def grpo_advantage_ex(rewards: torch.Tensor, G: int, mode: int = GRPO_ADV_DR, std_eps: float = 0.0,
                      adv=None, count_contrast: bool = False, stream=None):
    """Group advantage with the original GRPO option (mode GRPO_ADV_STD) and,
    if asked, the number of groups with reward contrast (an int32 device
    tensor).  Returns ``(adv, n_contrast or None)``."""
    _dev(rewards, "rewards", torch.float32)
    if adv is None:
        adv = torch.empty_like(rewards)
    n = rewards.numel()
    if G < 1 or n % G:
        raise ValueError("len(rewards) must be a multiple of G >= 1")
    cnt = torch.empty((1,), dtype=torch.int32, device=rewards.device) if count_contrast else None
    _check(_lib.grpo_advantage_ex(_ptr(rewards), n // G, G, int(mode), float(std_eps), _ptr(adv),
                                  _ptr(cnt), _stream(stream)), "grpo_advantage_ex")
    return adv, cnt


def grpo_workspace_size(N: int, C: int, V: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.grpo_workspace_size(N, C, V, ctypes.byref(out)), "grpo_workspace_size")
    return int(out.value)


def grpo_loss_fwd(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2,
                  beta=0.0, norm=0.0, out=None, workspace=None, stream=None, agg=None):
    """Per-token log-probs, gradient weights and the Dr. GRPO loss.

    ``logits`` [N, P+C, V] float32/bfloat16.  Returns a dict with ``logp``,
    ``lse``, ``w`` ([N, C] float32), ``loss`` (one-element float32 tensor on
    the device) and ``workspace``.  Pass ``out``/``workspace`` (as returned
    by an earlier call) to reuse buffers."""
    _dev(logits, "logits")
    N, T, V = logits.shape
    C = T - P
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("adv", adv, torch.float32), ("old_logp", old_logp, torch.float32),
                        ("ref_logp", ref_logp, torch.float32)):
        _dev(t, name, dt)
    dev = logits.device
    if out is None:
        out = {"logp": torch.empty((N, C), dtype=torch.float32, device=dev),
               "lse": torch.empty((N, C), dtype=torch.float32, device=dev),
               "w": torch.empty((N, C), dtype=torch.float32, device=dev),
               "loss": torch.empty((1,), dtype=torch.float32, device=dev)}
    need = grpo_workspace_size(N, C, V)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    out["workspace"] = workspace
    head = (_ptr(logits), _dtype_code(logits), N, P, C, V, _ptr(input_ids), _ptr(lens), _ptr(adv),
            _ptr(old_logp), _ptr(ref_logp), float(eps), float(beta), float(norm))
    tail = (_ptr(out["logp"]), _ptr(out["lse"]), _ptr(out["w"]), _ptr(out["loss"]),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if agg is None:
        _check(_lib.grpo_loss_fwd(*head, *tail), "grpo_loss_fwd")
    else:
        _check(_lib.grpo_loss_fwd_ex(*head, int(agg), *tail), "grpo_loss_fwd_ex")
    return out


def grpo_loss_fwd_ex(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2,
                     beta=0.0, norm=0.0, agg=GRPO_AGG_TOKEN_SUM, out=None, workspace=None,
                     stream=None):
    """grpo_loss_fwd with the aggregation choice (GRPO_AGG_TOKEN_SUM or
    GRPO_AGG_SEQ_MEAN)."""
    return grpo_loss_fwd(logits, P, input_ids, lens, adv, old_logp, ref_logp, eps, beta, norm,
                         out, workspace, stream, agg=agg)


def grpo_logprobs(logits, P, input_ids, lens, out=None, workspace=None, stream=None):
    """Log-probs only (the no-grad old/reference passes): ``(logp, lse,
    workspace)``, [N, C] float32, 0 past each length."""
    _dev(logits, "logits")
    N, T, V = logits.shape
    C = T - P
    _dev(input_ids, "input_ids", torch.int64)
    _dev(lens, "lens", torch.int32)
    dev = logits.device
    if out is None:
        out = (torch.empty((N, C), dtype=torch.float32, device=dev),
               torch.empty((N, C), dtype=torch.float32, device=dev))
    need = grpo_workspace_size(N, C, V)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    _check(_lib.grpo_logprobs(_ptr(logits), _dtype_code(logits), N, P, C, V, _ptr(input_ids),
                              _ptr(lens), _ptr(out[0]), _ptr(out[1]), _ptr(workspace),
                              workspace.numel(), _stream(stream)), "grpo_logprobs")
    return out[0], out[1], workspace


def grpo_loss_fwd_static(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None,
                         eps=0.2, beta=0.0, norm=0.0, out=None, stream=None):
    """grpo_loss_fwd using the library's built-in scratch instead of a
    caller-provided workspace (for callers that cannot allocate device
    memory).  Returns ``logp``, ``lse``, ``w`` and ``loss`` like
    :func:`grpo_loss_fwd`; ``out`` must be passed preallocated by a caller
    that cannot allocate."""
    _dev(logits, "logits")
    N, T, V = logits.shape
    C = T - P
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("adv", adv, torch.float32), ("old_logp", old_logp, torch.float32),
                        ("ref_logp", ref_logp, torch.float32)):
        _dev(t, name, dt)
    dev = logits.device
    if out is None:
        out = {"logp": torch.empty((N, C), dtype=torch.float32, device=dev),
               "lse": torch.empty((N, C), dtype=torch.float32, device=dev),
               "w": torch.empty((N, C), dtype=torch.float32, device=dev),
               "loss": torch.empty((1,), dtype=torch.float32, device=dev)}
    _check(_lib.grpo_loss_fwd_static(
        _ptr(logits), _dtype_code(logits), N, P, C, V, _ptr(input_ids), _ptr(lens), _ptr(adv),
        _ptr(old_logp), _ptr(ref_logp), float(eps), float(beta), float(norm), _ptr(out["logp"]),
        _ptr(out["lse"]), _ptr(out["w"]), _ptr(out["loss"]), _stream(stream)),
        "grpo_loss_fwd_static")
    return out


def grpo_loss_bwd(logits, P, input_ids, lens, lse, w, grad_loss=None, dlogits=None,
                  stream=None, flags=None):
    """d (grad_loss * loss) / d logits, same shape and dtype as ``logits``."""
    _dev(logits, "logits")
    N, T, V = logits.shape
    C = T - P
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("lse", lse, torch.float32), ("w", w, torch.float32),
                        ("grad_loss", grad_loss, torch.float32)):
        _dev(t, name, dt)
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    _dev(dlogits, "dlogits", logits.dtype)
    args = (_ptr(logits), _dtype_code(logits), N, P, C, V, _ptr(input_ids), _ptr(lens), _ptr(lse),
            _ptr(w), _ptr(grad_loss), _ptr(dlogits))
    if flags is None:
        _check(_lib.grpo_loss_bwd(*args, _stream(stream)), "grpo_loss_bwd")
    else:
        _check(_lib.grpo_loss_bwd_ex(*args, int(flags), _stream(stream)), "grpo_loss_bwd_ex")
    return dlogits


def grpo_loss_bwd_ex(logits, P, input_ids, lens, lse, w, grad_loss=None, dlogits=None, flags=0,
                     stream=None):
    """grpo_loss_bwd with flags (GRPO_BWD_SKIP_ZERO_WEIGHT)."""
    return grpo_loss_bwd(logits, P, input_ids, lens, lse, w, grad_loss, dlogits, stream, flags)


def grpo_loss_fwd_bwd(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2,
                      beta=0.0, norm=0.0, grad_loss=None, out=None, workspace=None,
                      dlogits=None, stream=None, agg=None):
    """Forward and backward in one pass over each scored row.  Returns the
    dict of :func:`grpo_loss_fwd` plus ``dlogits``."""
    _dev(logits, "logits")
    N, T, V = logits.shape
    C = T - P
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("adv", adv, torch.float32), ("old_logp", old_logp, torch.float32),
                        ("ref_logp", ref_logp, torch.float32),
                        ("grad_loss", grad_loss, torch.float32)):
        _dev(t, name, dt)
    dev = logits.device
    if out is None:
        out = {"logp": torch.empty((N, C), dtype=torch.float32, device=dev),
               "lse": torch.empty((N, C), dtype=torch.float32, device=dev),
               "w": torch.empty((N, C), dtype=torch.float32, device=dev),
               "loss": torch.empty((1,), dtype=torch.float32, device=dev)}
    need = grpo_workspace_size(N, C, V)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    _dev(dlogits, "dlogits", logits.dtype)
    out["workspace"] = workspace
    out["dlogits"] = dlogits
    head = (_ptr(logits), _dtype_code(logits), N, P, C, V, _ptr(input_ids), _ptr(lens), _ptr(adv),
            _ptr(old_logp), _ptr(ref_logp), float(eps), float(beta), float(norm))
    tail = (_ptr(grad_loss), _ptr(out["logp"]), _ptr(out["lse"]), _ptr(out["w"]),
            _ptr(out["loss"]), _ptr(dlogits), _ptr(workspace), workspace.numel(), _stream(stream))
    if agg is None:
        _check(_lib.grpo_loss_fwd_bwd(*head, *tail), "grpo_loss_fwd_bwd")
    else:
        _check(_lib.grpo_loss_fwd_bwd_ex(*head, int(agg), *tail), "grpo_loss_fwd_bwd_ex")
    return out


def grpo_loss_fwd_bwd_host(host_logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None,
                           eps=0.2, beta=0.0, norm=0.0, grad_loss=None, out=None, workspace=None,
                           dlogits=None, staging=None, stream=None):
    """:func:`grpo_loss_fwd_bwd` for logits in page-locked host memory
    (``host_logits`` a pinned CPU tensor): only the scored rows cross the
    host link, into the same rows of ``staging`` (a device tensor of the
    logits' shape, allocated when None).  ``dlogits`` may be a device tensor
    or a pinned CPU tensor (the kernels then write the gradient across the
    host link).  Returns the dict of :func:`grpo_loss_fwd_bwd` plus
    ``staging``."""
    if host_logits.is_cuda or not host_logits.is_pinned() or not host_logits.is_contiguous():
        raise ValueError("host_logits must be a contiguous pinned CPU tensor")
    N, T, V = host_logits.shape
    C = T - P
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("adv", adv, torch.float32), ("old_logp", old_logp, torch.float32),
                        ("ref_logp", ref_logp, torch.float32),
                        ("grad_loss", grad_loss, torch.float32)):
        _dev(t, name, dt)
    dev = input_ids.device
    if out is None:
        out = {"logp": torch.empty((N, C), dtype=torch.float32, device=dev),
               "lse": torch.empty((N, C), dtype=torch.float32, device=dev),
               "w": torch.empty((N, C), dtype=torch.float32, device=dev),
               "loss": torch.empty((1,), dtype=torch.float32, device=dev)}
    need = grpo_workspace_size(N, C, V)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if dlogits is None:
        dlogits = torch.empty(host_logits.shape, dtype=host_logits.dtype, device=dev)
    if staging is None:
        staging = torch.empty(host_logits.shape, dtype=host_logits.dtype, device=dev)
    if dlogits.is_cuda:
        _dev(dlogits, "dlogits", host_logits.dtype)
    elif (not dlogits.is_pinned() or not dlogits.is_contiguous()
          or dlogits.dtype != host_logits.dtype or dlogits.shape != host_logits.shape):
        raise ValueError("dlogits must be a CUDA tensor or a contiguous pinned CPU tensor of "
                         "the logits' shape and dtype")
    _dev(staging, "staging", host_logits.dtype)
    out.update(workspace=workspace, dlogits=dlogits, staging=staging)
    _check(_lib.grpo_loss_fwd_bwd_host(
        _ptr(host_logits), _dtype_code(host_logits), N, P, C, V, _ptr(input_ids), _ptr(lens),
        _ptr(adv), _ptr(old_logp), _ptr(ref_logp), float(eps), float(beta), float(norm),
        _ptr(grad_loss), _ptr(out["logp"]), _ptr(out["lse"]), _ptr(out["w"]), _ptr(out["loss"]),
        _ptr(dlogits), _ptr(staging), _ptr(workspace), workspace.numel(), _stream(stream)),
        "grpo_loss_fwd_bwd_host")
    return out


def grpo_loss_fwd_bwd_ex(logits, P, input_ids, lens, adv, old_logp=None, ref_logp=None, eps=0.2,
                         beta=0.0, norm=0.0, agg=GRPO_AGG_TOKEN_SUM, grad_loss=None, out=None,
                         workspace=None, dlogits=None, stream=None):
    """grpo_loss_fwd_bwd with the aggregation choice."""
    return grpo_loss_fwd_bwd(logits, P, input_ids, lens, adv, old_logp, ref_logp, eps, beta, norm,
                             grad_loss, out, workspace, dlogits, stream, agg=agg)


def grpo_lmhead_logprobs(hidden, weight, P, input_ids, lens, out=None, workspace=None,
                         stream=None):
    """Log-probs from hidden states [N, P+C, d] and the LM head [V, d] (both
    bfloat16), with the projection fused on the tensor cores.  Returns
    ``(logp, lse, workspace)``."""
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(weight, "weight", torch.bfloat16)
    _dev(input_ids, "input_ids", torch.int64)
    _dev(lens, "lens", torch.int32)
    N, T, d = hidden.shape
    V = weight.shape[0]
    C = T - P
    if weight.shape[1] != d:
        raise ValueError("weight must be [V, d]")
    dev = hidden.device
    if out is None:
        out = (torch.empty((N, C), dtype=torch.float32, device=dev),
               torch.empty((N, C), dtype=torch.float32, device=dev))
    need = ctypes.c_size_t(0)
    _check(_lib.grpo_lmhead_workspace_size(N, C, V, d, ctypes.byref(need)),
           "grpo_lmhead_workspace_size")
    if workspace is None or workspace.numel() < need.value:
        workspace = torch.empty((need.value,), dtype=torch.uint8, device=dev)
    _check(_lib.grpo_lmhead_logprobs(_ptr(hidden), _ptr(weight), N, P, C, V, d, _ptr(input_ids),
                                     _ptr(lens), _ptr(out[0]), _ptr(out[1]), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "grpo_lmhead_logprobs")
    return out[0], out[1], workspace


def grpo_lmhead_loss_fwd(hidden, weight, P, input_ids, lens, adv, old_logp=None, ref_logp=None,
                         eps=0.2, beta=0.0, norm=0.0, out=None, workspace=None, stream=None,
                         agg=None):
    """The Dr. GRPO loss forward from hidden states [N, P+C, d] and the LM
    head [V, d] (both bfloat16): the projection fused with the log-softmax on
    the tensor cores, then the surrogate.  Returns a dict like
    :func:`grpo_loss_fwd` (``logp``, ``lse``, ``w``, ``loss``, ``workspace``)."""
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(weight, "weight", torch.bfloat16)
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("adv", adv, torch.float32), ("old_logp", old_logp, torch.float32),
                        ("ref_logp", ref_logp, torch.float32)):
        _dev(t, name, dt)
    N, T, d = hidden.shape
    V = weight.shape[0]
    C = T - P
    if weight.shape[1] != d:
        raise ValueError("weight must be [V, d]")
    dev = hidden.device
    if out is None:
        out = {k: torch.empty((N, C), dtype=torch.float32, device=dev) for k in ("logp", "lse", "w")}
        out["loss"] = torch.empty((1,), dtype=torch.float32, device=dev)
    need = ctypes.c_size_t(0)
    _check(_lib.grpo_lmhead_workspace_size(N, C, V, d, ctypes.byref(need)),
           "grpo_lmhead_workspace_size")
    if workspace is None or workspace.numel() < need.value:
        workspace = torch.empty((need.value,), dtype=torch.uint8, device=dev)
    out["workspace"] = workspace
    head = (_ptr(hidden), _ptr(weight), N, P, C, V, d, _ptr(input_ids), _ptr(lens), _ptr(adv),
            _ptr(old_logp), _ptr(ref_logp), float(eps), float(beta), float(norm))
    tail = (_ptr(out["logp"]), _ptr(out["lse"]), _ptr(out["w"]), _ptr(out["loss"]),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if agg is None:
        _check(_lib.grpo_lmhead_loss_fwd(*head, *tail), "grpo_lmhead_loss_fwd")
    else:
        _check(_lib.grpo_lmhead_loss_fwd_ex(*head, int(agg), *tail), "grpo_lmhead_loss_fwd_ex")
    return out


def grpo_lmhead_bwd_workspace_size(N: int, C: int, V: int, d: int, rows_per_pass: int = 0) -> int:
    """Bytes of the LM-head backward's workspace for passes of
    ``rows_per_pass`` backward rows (0: one pass over all N*C)."""
    out = ctypes.c_size_t(0)
    _check(_lib.grpo_lmhead_bwd_workspace_size_rows(N, C, V, d, int(rows_per_pass),
                                                    ctypes.byref(out)),
           "grpo_lmhead_bwd_workspace_size_rows")
    return int(out.value)


def grpo_lmhead_loss_bwd(hidden, weight, P, input_ids, lens, lse, w, grad_loss=None, out=None,
                         workspace=None, stream=None, flags=None, rows_per_pass=0):
    """Gradients of ``grad_loss * loss`` with respect to the hidden states and
    the LM head.  Returns ``(dhidden [N, P+C, d], dweight [V, d], workspace)``,
    float32; ``out`` = (dhidden, dweight) to reuse buffers.  Without a
    ``workspace`` one is allocated for passes of ``rows_per_pass`` rows (0:
    one pass over every possible row); a given workspace sets the passes by
    its size."""
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(weight, "weight", torch.bfloat16)
    for name, t, dt in (("input_ids", input_ids, torch.int64), ("lens", lens, torch.int32),
                        ("lse", lse, torch.float32), ("w", w, torch.float32),
                        ("grad_loss", grad_loss, torch.float32)):
        _dev(t, name, dt)
    N, T, d = hidden.shape
    V = weight.shape[0]
    C = T - P
    dev = hidden.device
    if out is None:
        out = (torch.empty((N, T, d), dtype=torch.float32, device=dev),
               torch.empty((V, d), dtype=torch.float32, device=dev))
    if workspace is None:
        need = grpo_lmhead_bwd_workspace_size(N, C, V, d, rows_per_pass)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    head = (_ptr(hidden), _ptr(weight), N, P, C, V, d, _ptr(input_ids), _ptr(lens), _ptr(lse),
            _ptr(w), _ptr(grad_loss), _ptr(out[0]), _ptr(out[1]))
    tail = (_ptr(workspace), workspace.numel(), _stream(stream))
    if flags is None:
        _check(_lib.grpo_lmhead_loss_bwd(*head, *tail), "grpo_lmhead_loss_bwd")
    else:
        _check(_lib.grpo_lmhead_loss_bwd_ex(*head, int(flags), *tail), "grpo_lmhead_loss_bwd_ex")
    return out[0], out[1], workspace


def grpo_set_early_start(enable: bool) -> None:
    """Turns the early starts of grpo_loss_bwd (after grpo_loss_fwd) and
    grpo_advantage (after grpo_mask) on or off for the process."""
    _lib.grpo_set_early_start(1 if enable else 0)


def grpo_selftest_timeout(workspace, stream=None) -> None:
    """Launches the bounded-wait self-test on ``workspace`` (a uint8 device
    tensor of at least 16 bytes, 256-byte aligned): about a second later its
    error flags hold a timeout, which grpo_check_error reports as
    GRPO_ERR_TIMEOUT (8)."""
    _dev(workspace, "workspace")
    _check(_lib.grpo_selftest_timeout(_ptr(workspace), _stream(stream)), "grpo_selftest_timeout")


def grpo_check_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the status the last forward call
    on ``workspace`` recorded (0 = GRPO_OK); does not raise."""
    return int(_lib.grpo_check_error(_ptr(workspace), _stream(stream)))


def grpo_copy(dst: torch.Tensor, src: torch.Tensor, nbytes: int | None = None, stream=None):
    """Vector device-to-device copy (the HBM copy ceiling)."""
    nbytes = src.numel() * src.element_size() if nbytes is None else nbytes
    _check(_lib.grpo_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "grpo_copy")
    return dst
