"""The C-ABI library loads, exports every symbol include/grpo.h declares, and
rejects invalid arguments on the host before any CUDA call.  CPU only: no
call here reaches a launch."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED, WORKSPACE, MISALIGNED = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    from vocab_wide_logprob_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    P, I64, F, SZ, INT = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t,
                          ctypes.c_int)
    lib.grpo_status_string.argtypes = [INT]
    lib.grpo_status_string.restype = ctypes.c_char_p
    lib.grpo_mask.argtypes = [P, I64, I64, I64, I64, P, P, P]
    lib.grpo_advantage.argtypes = [P, I64, I64, P, P]
    lib.grpo_workspace_size.argtypes = [I64, I64, I64, ctypes.POINTER(SZ)]
    lib.grpo_loss_fwd.argtypes = [P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, P, P, P, P,
                                  P, SZ, P]
    lib.grpo_loss_bwd.argtypes = [P, INT, I64, I64, I64, I64, P, P, P, P, P, P, P]
    lib.grpo_check_error.argtypes = [P, P]
    lib.grpo_copy.argtypes = [P, P, SZ, P]
    lib.grpo_lmhead_logprobs.argtypes = [P, P, I64, I64, I64, I64, I64, P, P, P, P, P, SZ, P]
    lib.grpo_advantage_ex.argtypes = [P, I64, I64, INT, F, P, P, P]
    lib.grpo_loss_bwd_ex.argtypes = [P, INT, I64, I64, I64, I64, P, P, P, P, P, P, ctypes.c_uint32, P]
    lib.grpo_loss_fwd_ex.argtypes = [P, INT, I64, I64, I64, I64, P, P, P, P, P, F, F, F, INT, P, P,
                                     P, P, P, SZ, P]
    return lib


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"^\w[\w\s\*]*?\b(grpo_\w+)\s*\(", src, re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("grpo_mask", "grpo_advantage", "grpo_loss_fwd", "grpo_loss_bwd",
              "grpo_workspace_size", "grpo_check_error"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(9):
        assert lib.grpo_status_string(code)
    assert lib.grpo_status_string(0) == b"ok"
    assert lib.grpo_status_string(99) == b"unknown status"


def A(addr):
    return ctypes.c_void_p(addr)


def test_mask_validation(lib):
    assert lib.grpo_mask(A(0x1000), -1, 4, 4, 2, None, A(0x2000), None) == INVALID
    assert lib.grpo_mask(A(0x1000), 2, -1, 4, 2, None, A(0x2000), None) == INVALID
    assert lib.grpo_mask(A(0x1000), 2, 4, 4, 2, None, None, None) == INVALID
    assert lib.grpo_mask(A(0x1004), 2, 4, 4, 2, None, A(0x2000), None) == MISALIGNED
    assert lib.grpo_mask(A(0x1000), 2, 4, 4, 2, None, A(0x2002), None) == MISALIGNED
    assert lib.grpo_mask(None, 0, 4, 4, 2, None, None, None) == OK  # nothing to do
    big = (1 << 63) - 1  # P + C would not fit in int64
    assert lib.grpo_mask(A(0x1000), 2, big, 4, 2, None, A(0x2000), None) == UNSUPPORTED


def test_advantage_validation(lib):
    assert lib.grpo_advantage(A(0x1000), 2, 0, A(0x2000), None) == INVALID
    assert lib.grpo_advantage(A(0x1000), -1, 4, A(0x2000), None) == INVALID
    assert lib.grpo_advantage(None, 2, 4, A(0x2000), None) == INVALID
    assert lib.grpo_advantage(A(0x1002), 2, 4, A(0x2000), None) == MISALIGNED
    assert lib.grpo_advantage(None, 0, 4, None, None) == OK


def test_workspace_size(lib):
    out = ctypes.c_size_t(0)
    assert lib.grpo_workspace_size(64, 1024, 151936, ctypes.byref(out)) == OK
    assert out.value % 256 == 0 and out.value >= 256 + 4 * 65 + 4 * 64 + 8 * 1024
    assert lib.grpo_workspace_size(-1, 4, 4, ctypes.byref(out)) == INVALID
    assert lib.grpo_workspace_size(1 << 20, 1 << 12, 4, ctypes.byref(out)) == UNSUPPORTED
    assert lib.grpo_workspace_size(4, 4, 4, None) == INVALID


def _fwd(lib, **kw):
    args = dict(logits=A(0x10000), dtype=1, N=8, P=4, C=8, V=64, ids=A(0x20000),
                len=A(0x30000), adv=A(0x40000), old=None, ref=None, eps=0.2, beta=0.0,
                norm=0.0, logp=A(0x50000), lse=A(0x60000), w=A(0x70000), loss=A(0x80000),
                ws=A(0x100000), ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.grpo_loss_fwd(*args.values())


def test_fwd_validation(lib):
    assert _fwd(lib, dtype=7) == UNSUPPORTED
    assert _fwd(lib, N=-1) == INVALID
    assert _fwd(lib, P=0) == INVALID          # token 0 needs logits row P-1
    assert _fwd(lib, V=0) == INVALID
    assert _fwd(lib, eps=1.0) == INVALID
    assert _fwd(lib, eps=-0.1) == INVALID
    assert _fwd(lib, eps=float("nan")) == INVALID
    assert _fwd(lib, beta=-1.0) == INVALID
    assert _fwd(lib, beta=0.04) == INVALID    # beta > 0 needs reference log-probs
    assert _fwd(lib, norm=float("inf")) == INVALID
    assert _fwd(lib, loss=None) == INVALID
    assert _fwd(lib, ws=None) == INVALID
    assert _fwd(lib, logits=None) == INVALID
    assert _fwd(lib, logits=A(0x10001)) == MISALIGNED
    assert _fwd(lib, ws=A(0x100010)) == MISALIGNED
    assert _fwd(lib, ids=A(0x20004)) == MISALIGNED
    assert _fwd(lib, ws_bytes=64) == WORKSPACE
    assert _fwd(lib, N=1 << 20, C=1 << 12) == UNSUPPORTED   # N*C >= 2^31
    assert _fwd(lib, P=(1 << 63) - 1) == UNSUPPORTED         # P + C would not fit in int64


def _bwd(lib, **kw):
    args = dict(logits=A(0x10000), dtype=1, N=8, P=4, C=8, V=64, ids=A(0x20000),
                len=A(0x30000), lse=A(0x40000), w=A(0x50000), grad=None,
                dlogits=A(0x10000000), stream=None)
    args.update(kw)
    return lib.grpo_loss_bwd(*args.values())


def test_bwd_validation(lib):
    assert _bwd(lib, dtype=3) == UNSUPPORTED
    assert _bwd(lib, dlogits=None) == INVALID
    assert _bwd(lib, P=0) == INVALID
    assert _bwd(lib, dlogits=A(0x10002)) == INVALID   # overlaps the logits
    assert _bwd(lib, dlogits=A(0x10000001)) == MISALIGNED
    assert _bwd(lib, grad=A(0x60001)) == MISALIGNED
    assert _bwd(lib, N=0, dlogits=None) == OK


def test_copy_validation(lib):
    assert lib.grpo_copy(A(0x1000), A(0x2008), 64, None) == MISALIGNED
    assert lib.grpo_copy(A(0x1000), A(0x2000), 40, None) == MISALIGNED
    assert lib.grpo_copy(A(0x1000), A(0x1010), 64, None) == INVALID   # overlap
    assert lib.grpo_copy(None, None, 0, None) == OK
    assert lib.grpo_check_error(None, None) == INVALID


def test_extended_entry_validation(lib):
    a = A(0x10000)
    # advantage modes and epsilon
    assert lib.grpo_advantage_ex(a, 2, 4, 7, 0.0, A(0x20000), None, None) == UNSUPPORTED
    assert lib.grpo_advantage_ex(a, 2, 4, 1, -1.0, A(0x20000), None, None) == INVALID
    assert lib.grpo_advantage_ex(a, 2, 4, 1, 0.0, A(0x20000), A(0x30002), None) == MISALIGNED
    # backward flags
    assert lib.grpo_loss_bwd_ex(a, 1, 8, 4, 8, 64, A(0x20000), A(0x30000), A(0x40000),
                                A(0x50000), None, A(0x10000000), 2, None) == UNSUPPORTED
    # aggregation
    assert lib.grpo_loss_fwd_ex(a, 1, 8, 4, 8, 64, A(0x20000), A(0x30000), A(0x40000), None, None,
                                0.2, 0.0, 0.0, 5, A(0x50000), A(0x60000), A(0x70000), A(0x80000),
                                A(0x100000), 1 << 20, None) == UNSUPPORTED
    # LM head: hidden size a multiple of 128, 16-byte aligned operands
    args = [a, A(0x200000), 8, 4, 8, 1000, 96, A(0x20000), A(0x30000), A(0x40000), A(0x50000),
            A(0x100000), 1 << 30, None]
    assert lib.grpo_lmhead_logprobs(*args) == UNSUPPORTED
    args[6] = 192
    assert lib.grpo_lmhead_logprobs(*args) == UNSUPPORTED
    args[6] = 128
    args[0] = A(0x10008)
    assert lib.grpo_lmhead_logprobs(*args) == MISALIGNED
    args[0] = a
    args[11] = None
    assert lib.grpo_lmhead_logprobs(*args) == INVALID
