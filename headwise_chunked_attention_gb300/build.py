"""Build libupipe.so (the C ABI of include/upipe.h) for sm_103a, in-tree.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
``headwise_chunked_attention_gb300/_build/libupipe.so``.  No cmake, no torch
extension machinery: the library has a plain C ABI.

``build(debug=True)`` builds the same sources with UPIPE_DEBUG_BOUNDS into
``_build_debug/libupipe.so``: every plain (non-TMA) global load and store in
the kernels is checked against the extent of its view, and a failed check
reports UPIPE_ERR_BOUNDS instead of touching memory.  The binding loads it
when UPIPE_DEBUG_BOUNDS=1 is set in the environment.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libupipe.so")
OUT_DEBUG = os.path.join(PKG, "_build_debug")
SOURCES = ["upipe.cu", "gemm.cu", "attn_fwd.cu", "attn_bwd.cu", "elementwise.cu", "noalloc.cu",
           "selftest.cu", "mlp.cu", "loss.cu", "offload.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in deps)


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile what is stale and link libupipe.so (``debug``: the bounds-
    checked build in _build_debug/).  Processes that build at the same time
    (one per rank under torchrun) take turns on a file lock, so no object
    file is written by two nvcc runs at once."""
    import fcntl
    out = OUT_DEBUG if debug else OUT
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, ".build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(verbose, force, out,
                                 ["-DUPIPE_DEBUG_BOUNDS"] if debug else [])
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(verbose: bool, force: bool, out: str, extra) -> str:
    lib = os.path.join(out, "libupipe.so")
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC)
               if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "upipe.h"))
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            jobs.append([cc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, res in zip(jobs, ex.map(
                lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            if verbose or res.returncode:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    objs = [os.path.join(out, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(lib, objs):
        cmd = [cc, *ARCH, "-shared", "-o", lib + ".tmp", *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("link failed")
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
