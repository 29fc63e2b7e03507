"""Build libliger.so (the C-ABI library) in-tree for sm_103a.

Each translation unit under csrc/ is compiled by nvcc in parallel, then
linked into ``transformer_rmsnorm_fwd_gb300/libliger.so``.  Run as a module
(``python -m transformer_rmsnorm_fwd_gb300.build``) or through
``__graft_entry__.build()``.  Incremental: a unit is recompiled when it or
any header is newer than its object.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libliger.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool) -> list:
    f = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr", "-Wno-deprecated-gpu-targets"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_time = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    cc = nvcc()
    flags = _flags(verbose_ptxas)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        if (not force and not verbose_ptxas and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time)):
            return obj, ""
        cmd = [cc, *flags, "-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stderr

    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for o, log in results:
            if log:
                sys.stderr.write(f"--- {os.path.basename(o)}\n{log}")
    lib_time = os.path.getmtime(LIB) if os.path.exists(LIB) else -1
    if force or lib_time < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        p = subprocess.run([cc, "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
