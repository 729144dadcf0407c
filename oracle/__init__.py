"""Float64 CPU oracle for the Dr. GRPO loss over policy logits.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this package.  The CUDA library
(``vocab_wide_logprob_gb300``) never imports it, and it imports nothing from
that library: the two share no code, header, table or constant.  The seeded
input generators (``vocab_wide_logprob_gb300.workloads``) are the one module
both sides use, and that module holds none of the method's arithmetic.

The arithmetic lives in ``grpo_oracle.c`` (plain C, IEEE double, no
fast-math, no FMA contraction); this module compiles it with gcc, loads it
with ctypes and marshals numpy arrays.  Each method cites the part of the page
"Making Dr GRPO go brrr" (salahadawi.com) that it restates:

* :meth:`Oracle.mask`       -- "The completion mask" (``build_completion_mask``)
* :meth:`Oracle.advantage`  -- "Dr. GRPO": A_i = R_i - group mean, no sigma
* :meth:`Oracle.contrast_count` -- the analysis page "The Quiet Library",
  "The sparse-reward bottleneck": groups whose rewards are not all equal
* :meth:`Oracle.logp`, :meth:`Oracle.logp_rows` -- "compute_logprobs": shift
  by one, ``log_softmax`` over the vocabulary, gather at the sampled id
* :meth:`Oracle.loss`       -- "The loss" (``grpo_loss``) plus the pseudo-code's
  ``beta * kl`` term (k3 estimator; the page does not print one) and token-sum
  aggregation over a constant normaliser
* :meth:`Oracle.dlogits`, :meth:`Oracle.dlogits_row` -- "loss.backward()": the
  gradient with respect to the logits (chain rule; the page prints none)
* :meth:`Oracle.lmhead_logp`, :meth:`Oracle.lmhead_grads` -- the same through
  the LM-head projection ``model(...).logits`` = hidden x W^T: log-probs from
  hidden states, and the gradients with respect to the hidden states and W

Logits are numpy arrays of ``float32`` (``"f32"``), ``float64`` (``"f64"``,
for finite differences) or ``uint16`` holding bfloat16 bit patterns
(``"bf16"``).

Pins: ``tests/test_oracle_pins.py`` checks every method against values the
pages print, closed forms, library routines and finite differences, and
``tests/test_oracle_mutants.py`` shows that planted mistakes fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "grpo_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

_DTYPES = {"f32": 0, "float32": 0, "bf16": 1, "bfloat16": 1, "f64": 2, "float64": 2}
_NP = {0: np.float32, 1: np.uint16, 2: np.float64}


def compile_source(src: str, out: str) -> str:
    """gcc -O2, IEEE double semantics (no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fno-fast-math", "-ffp-contract=off",
           "-Wall", "-shared", "-fPIC", src, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``grpo_oracle.c`` into ``liboracle.so`` beside it (if stale)."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    return compile_source(SOURCE, LIBRARY)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc == -2:
        raise ValueError(f"{what}: a sampled token id is outside [0, V)")
    if rc != 0:
        raise ValueError(f"{what}: invalid arguments (code {rc})")


def _logits_arg(x, dtype):
    code = _DTYPES.get(dtype)
    if code is None:
        raise ValueError(f"unsupported logits dtype {dtype!r}")
    x = np.ascontiguousarray(x)
    if x.dtype != _NP[code]:
        raise TypeError(f"{dtype} logits must be a {np.dtype(_NP[code]).name} array")
    return x, code


def _wide(x):
    """float64 copy of a float array or of uint16 bfloat16 bit patterns (exact)."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


class Oracle:
    """One loaded build of the oracle library."""

    _SIG = None

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P, I64, D, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        sig = {
            "oracle_mask": [P, I64, I64, I64, I64, P, P],
            "oracle_advantage": [P, I64, I64, P],
            "oracle_advantage_std": [P, I64, I64, D, P],
            "oracle_contrast_count": [P, I64, I64, P],
            "oracle_loss_agg": [P, P, P, P, P, I64, I64, D, D, D, INT, P, P, P],
            "oracle_logp_rows": [P, INT, I64, I64, P, P, P],
            "oracle_logp": [P, INT, I64, I64, I64, I64, P, P, P, P],
            "oracle_loss": [P, P, P, P, P, I64, I64, D, D, D, P, P, P],
            "oracle_dlogits_row": [P, INT, I64, I64, D, D, P],
            "oracle_dlogits": [P, INT, I64, I64, I64, I64, P, P, P, P, D, P],
            "oracle_set_threads": [INT],
            "oracle_get_threads": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = None if name == "oracle_set_threads" else INT
        self.lib = lib
        self.path = path

    # -- threads ------------------------------------------------------------
    def set_threads(self, n: int) -> None:
        """POSIX threads for the row loops (0 = one per online core)."""
        self.lib.oracle_set_threads(int(n))

    def threads(self) -> int:
        return int(self.lib.oracle_get_threads())

    # -- "The completion mask" ---------------------------------------------
    def mask(self, ids: np.ndarray, P: int, C: int, eos_id: int):
        """Mask of ``ids`` [N, P+C] (int64) -> ``(mask u8 [N, C], len i32 [N])``:
        1 up to and including the first EOS of the completion, 0 after it,
        all 1 when the completion holds no EOS."""
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        if ids.ndim != 2 or ids.shape[1] != P + C:
            raise ValueError("ids must be [N, P + C]")
        N = ids.shape[0]
        m = np.zeros((N, C), np.uint8)
        ln = np.zeros(N, np.int32)
        _check(self.lib.oracle_mask(_ptr(ids), N, P, C, int(eos_id), _ptr(m), _ptr(ln)), "mask")
        return m, ln

    # -- "Dr. GRPO" advantage ----------------------------------------------
    def advantage(self, rewards: np.ndarray, G: int) -> np.ndarray:
        """A_i = R_i - mean of its group of G consecutive completions (double)."""
        R = np.ascontiguousarray(rewards, dtype=np.float64).reshape(-1)
        if G < 1 or R.size % G:
            raise ValueError("len(rewards) must be a multiple of G >= 1")
        A = np.zeros_like(R)
        _check(self.lib.oracle_advantage(_ptr(R), R.size // G, G, _ptr(A)), "advantage")
        return A

    def advantage_std(self, rewards: np.ndarray, G: int, std_eps: float = 0.0) -> np.ndarray:
        """Original GRPO: A_i = (R_i - mean) / (std + std_eps) within the group
        (std over the G rewards, dividing by G)."""
        R = np.ascontiguousarray(rewards, dtype=np.float64).reshape(-1)
        if G < 1 or R.size % G:
            raise ValueError("len(rewards) must be a multiple of G >= 1")
        A = np.zeros_like(R)
        _check(self.lib.oracle_advantage_std(_ptr(R), R.size // G, G, float(std_eps), _ptr(A)),
               "advantage_std")
        return A

    # -- "The sparse-reward bottleneck" ----------------------------------------
    def contrast_count(self, rewards: np.ndarray, G: int) -> int:
        """Number of groups of G consecutive completions whose rewards are not
        all equal (the groups that carry a learning signal; a uniform group's
        advantages are all zero)."""
        R = np.ascontiguousarray(rewards, dtype=np.float64).reshape(-1)
        if G < 1 or R.size % G:
            raise ValueError("len(rewards) must be a multiple of G >= 1")
        out = ctypes.c_int64(0)
        _check(self.lib.oracle_contrast_count(_ptr(R), R.size // G, G, ctypes.addressof(out)),
               "contrast_count")
        return int(out.value)

    # -- "compute_logprobs" --------------------------------------------------
    def logp_rows(self, rows: np.ndarray, dtype: str, y: np.ndarray):
        """Independent rows [n, V] -> ``(logp [n], lse [n])``,
        logp = z[y] - logsumexp(z)."""
        rows, code = _logits_arg(rows, dtype)
        n, V = rows.shape
        y = np.ascontiguousarray(y, dtype=np.int64).reshape(n)
        lp = np.zeros(n)
        ls = np.zeros(n)
        _check(self.lib.oracle_logp_rows(_ptr(rows), code, n, V, _ptr(y), _ptr(lp), _ptr(ls)),
               "logp_rows")
        return lp, ls

    def logp(self, logits: np.ndarray, dtype: str, P: int, C: int, ids, lens):
        """Batch: logits [N, P+C, V], ids [N, P+C], lens [N] -> ``(logp, lse)``
        [N, C] in double, 0 past each length.  Token t of completion i is
        scored by logits row P-1+t."""
        logits, code = _logits_arg(logits, dtype)
        N, T, V = logits.shape
        if T != P + C:
            raise ValueError("logits must be [N, P + C, V]")
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        lp = np.zeros((N, C))
        ls = np.zeros((N, C))
        _check(self.lib.oracle_logp(_ptr(logits), code, N, P, C, V, _ptr(ids), _ptr(lens),
                                    _ptr(lp), _ptr(ls)), "logp")
        return lp, ls

    def lmhead_logp(self, hidden, weight, P: int, C: int, ids, lens):
        """Log-probs from hidden states [N, P+C, d] and the LM head [V, d]
        ("model(...).logits" = hidden x W^T, then "compute_logprobs"): the
        scored rows' logits in float64 (numpy matmul of the exactly widened
        bf16 inputs), then :meth:`logp_rows`.  Inputs are uint16 bf16 bit
        patterns or float arrays.  Returns ``(logp, lse)`` [N, C]."""
        H = _wide(hidden)
        W = _wide(weight)
        N = H.shape[0]
        ids = np.asarray(ids, dtype=np.int64)
        lens = np.asarray(lens, dtype=np.int32)
        lp = np.zeros((N, C))
        ls = np.zeros((N, C))
        for i in range(N):
            L = int(lens[i])
            if L == 0:
                continue
            z = H[i, P - 1:P - 1 + L] @ W.T
            a, b = self.logp_rows(z, "f64", ids[i, P:P + L])
            lp[i, :L] = a
            ls[i, :L] = b
        return lp, ls

    def lmhead_grads(self, hidden, weight, P: int, C: int, ids, lens, lse, w, g: float = 1.0,
                     rows=None, vocab=None, magnitudes: bool = False):
        """Gradients of ``g * loss`` through the LM head ("loss.backward()" of
        the loss over ``model(...).logits`` = hidden x W^T): each scored row's
        logits gradient dz from :meth:`dlogits_row` (lse and w as the forward
        left them), then by the chain rule through z = h W^T
        dhidden[i, P-1+t] = dz W and dweight = sum over scored rows of dz^T h
        (numpy float64 matmuls of the exactly widened inputs).  Rows that score
        nothing get a zero dhidden.

        ``rows``: None for the whole dhidden [N, P+C, d], or a list of
        completion positions (i, t) for just those rows ([len(rows), d];
        positions that score nothing give zero rows).  ``vocab``: None for the
        whole dweight [V, d], or vocabulary ids for just those rows.
        ``magnitudes``: also return |dz| |W| and |dz|^T |h| with the same
        shapes (the sums whose terms a rounding of dz perturbs).
        Returns ``dict(dhidden=..., dweight=...[, dhidden_mag=..., dweight_mag=...])``."""
        H = _wide(hidden)
        W = _wide(weight)
        N, T, d = H.shape
        V = W.shape[0]
        ids = np.asarray(ids, dtype=np.int64)
        lens = np.asarray(lens, dtype=np.int32)
        lse = np.asarray(lse, dtype=np.float64)
        w = np.asarray(w, dtype=np.float64)
        vsel = np.arange(V) if vocab is None else np.asarray(vocab, dtype=np.int64)
        dH = np.zeros((N, T, d) if rows is None else (len(rows), d))
        dW = np.zeros((len(vsel), d))
        mH = np.zeros_like(dH) if magnitudes else None
        mW = np.zeros_like(dW) if magnitudes else None
        absW = np.abs(W) if magnitudes else None
        for i in range(N):
            L = int(lens[i])
            if L == 0:
                continue
            h = H[i, P - 1:P - 1 + L]           # the rows that score tokens 0..L-1
            z = h @ W.T
            dz = np.stack([self.dlogits_row(z[t], "f64", int(ids[i, P + t]), lse[i, t],
                                            g * w[i, t]) for t in range(L)])
            if rows is None:
                dH[i, P - 1:P - 1 + L] = dz @ W
                if magnitudes:
                    mH[i, P - 1:P - 1 + L] = np.abs(dz) @ absW
            else:
                for k, (ii, t) in enumerate(rows):
                    if ii == i and 0 <= t < L:
                        dH[k] = dz[t] @ W
                        if magnitudes:
                            mH[k] = np.abs(dz[t]) @ absW
            dzs = dz[:, vsel]
            dW += dzs.T @ h
            if magnitudes:
                mW += np.abs(dzs).T @ np.abs(h)
        out = dict(dhidden=dH, dweight=dW)
        if magnitudes:
            out.update(dhidden_mag=mH, dweight_mag=mW)
        return out

    # -- "The loss" ------------------------------------------------------------
    def loss_seq_mean(self, logp, old, ref, adv, lens, eps: float, beta: float,
                      norm: float = 0.0):
        """Original GRPO aggregation: each completion's token sum divided by its
        length, summed over completions and divided by ``norm`` (<= 0: N).
        Returns ``(loss, w, ell)`` like :meth:`loss`."""
        return self._loss(logp, old, ref, adv, lens, eps, beta, norm, 1)

    def loss(self, logp, old, ref, adv, lens, eps: float, beta: float, norm: float = 0.0):
        """Dr. GRPO loss.  ``old=None``: old log-probs equal current ones
        (ratio exactly 1).  ``ref`` may be None only when beta == 0.
        ``norm <= 0`` selects N*C.  Returns ``(loss, w [N, C], ell [N, C])``,
        ell the per-token loss and w = d loss / d logp."""
        return self._loss(logp, old, ref, adv, lens, eps, beta, norm, 0)

    def _loss(self, logp, old, ref, adv, lens, eps, beta, norm, agg):
        lp = np.ascontiguousarray(logp, dtype=np.float64)
        N, C = lp.shape
        old = None if old is None else np.ascontiguousarray(old, dtype=np.float64)
        ref = None if ref is None else np.ascontiguousarray(ref, dtype=np.float64)
        A = np.ascontiguousarray(adv, dtype=np.float64).reshape(N)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        out = ctypes.c_double(0.0)
        w = np.zeros((N, C))
        ell = np.zeros((N, C))
        _check(self.lib.oracle_loss_agg(_ptr(lp), _ptr(old), _ptr(ref), _ptr(A), _ptr(lens), N, C,
                                        float(eps), float(beta), float(norm), int(agg),
                                        ctypes.addressof(out), _ptr(w), _ptr(ell)), "loss")
        return out.value, w, ell

    # -- "loss.backward()" -----------------------------------------------------
    def dlogits_row(self, row: np.ndarray, dtype: str, y: int, lse: float, gw: float):
        """One scored row: gw * (onehot(y) - softmax(row)), in double."""
        row, code = _logits_arg(row, dtype)
        out = np.zeros(row.shape[-1])
        _check(self.lib.oracle_dlogits_row(_ptr(row), code, row.shape[-1], int(y), float(lse),
                                           float(gw), _ptr(out)), "dlogits_row")
        return out

    def dlogits(self, logits, dtype: str, P: int, C: int, ids, lens, lse, w, g: float = 1.0):
        """d (g * loss) / d logits over the whole [N, P+C, V] batch (double);
        rows that score no valid completion token are 0."""
        logits, code = _logits_arg(logits, dtype)
        N, T, V = logits.shape
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        lse = np.ascontiguousarray(lse, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        out = np.zeros((N, T, V))
        _check(self.lib.oracle_dlogits(_ptr(logits), code, N, P, C, V, _ptr(ids), _ptr(lens),
                                       _ptr(lse), _ptr(w), float(g), _ptr(out)), "dlogits")
        return out


_lock = threading.Lock()
_default = None


def default() -> Oracle:
    """The oracle built from ``grpo_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def mask(*a, **k):
    return default().mask(*a, **k)


def advantage(*a, **k):
    return default().advantage(*a, **k)


def advantage_std(*a, **k):
    return default().advantage_std(*a, **k)


def contrast_count(*a, **k):
    return default().contrast_count(*a, **k)


def loss_seq_mean(*a, **k):
    return default().loss_seq_mean(*a, **k)


def logp_rows(*a, **k):
    return default().logp_rows(*a, **k)


def logp(*a, **k):
    return default().logp(*a, **k)


def loss(*a, **k):
    return default().loss(*a, **k)


def lmhead_logp(*a, **k):
    return default().lmhead_logp(*a, **k)


def lmhead_grads(*a, **k):
    return default().lmhead_grads(*a, **k)


def dlogits_row(*a, **k):
    return default().dlogits_row(*a, **k)


def dlogits(*a, **k):
    return default().dlogits(*a, **k)


def set_threads(n: int) -> None:
    default().set_threads(n)


def threads() -> int:
    return default().threads()
