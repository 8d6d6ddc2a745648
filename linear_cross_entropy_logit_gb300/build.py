"""Build the in-tree CUDA library ``_lib/libflce.so`` for sm_103a with nvcc.

Usage: ``python -m linear_cross_entropy_logit_gb300.build [--force] [--verbose]``.
Each translation unit is compiled in parallel to an object file under
``_build/``, then linked.  The library is rebuilt when any source under
``csrc/`` or the public header is newer than the built file.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(LIBDIR, "libflce.so")
SOURCES = ["flce_api.cu", "flce_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflce")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "flce.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(OBJDIR, exist_ok=True)
    tag = os.getpid()
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(OBJDIR, f"{os.path.splitext(src)[0]}.{tag}.o")
        cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
               "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                            text=True)))
        objs.append(obj)
    failed = False
    for src, p in procs:
        out, err = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out)
            sys.stderr.write(err)
        if p.returncode != 0:
            print(f"nvcc failed on {src} (exit {p.returncode})", file=sys.stderr)
            failed = True
    if failed:
        raise RuntimeError("nvcc compilation failed")
    tmp = LIB + f".tmp{tag}"
    link = [nvcc(), *ARCH, "-shared", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stdout.write(r.stdout)
        sys.stderr.write(r.stderr)
    for o in objs:
        try:
            os.remove(o)
        except OSError:
            pass
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed with exit code {r.returncode}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
          ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)
