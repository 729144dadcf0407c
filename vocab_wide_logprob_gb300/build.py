"""Builds ``libgrpo.so`` (the C-ABI CUDA library) in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in ``_build/`` in parallel,
then linked into ``vocab_wide_logprob_gb300/libgrpo.so`` against the shared
CUDA runtime (so the process keeps a single runtime instance with PyTorch).
Run as ``python -m vocab_wide_logprob_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(PKG, "libgrpo.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def compile_flags(verbose_ptxas: bool = False):
    flags = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
             "-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def _compile(src: str, verbose_ptxas: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if verbose_ptxas or _stale(obj, [src, *_headers()]):
        cmd = [nvcc(), *compile_flags(verbose_ptxas), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr
    return obj, ""


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    """Compiles the library if any source is newer than it; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas and not quiet:
        for _, log in results:
            sys.stderr.write(log)
    if force or _stale(LIBRARY, objs):
        tmp = LIBRARY + f".tmp{os.getpid()}"
        lib64 = os.path.join(cuda_home(), "lib64")
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", f"-rpath,{lib64}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force="--force" in sys.argv, verbose_ptxas=v, quiet=not v))
