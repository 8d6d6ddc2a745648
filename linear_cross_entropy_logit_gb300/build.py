"""Build the in-tree CUDA libraries for sm_103a with nvcc.

  _lib/libflce.so        the library
  _lib/libflce_debug.so  the same sources compiled with FLCE_DEBUG: the
                         device-side index math (tile lists, row bands, skip
                         lists, filter masks, partial slots) is range-checked
                         and an out-of-range index sets FLCE_ERR_BOUNDS in the
                         error word instead of being used

Usage: ``python -m linear_cross_entropy_logit_gb300.build [--force] [--verbose]``.
Every translation unit of both libraries is compiled in parallel to an object
file under ``_build/``, then each library is linked.  A library is rebuilt when
any source under ``csrc/`` or the public header is newer than it.
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
DEBUG_LIB = os.path.join(LIBDIR, "libflce_debug.so")
SOURCES = ["flce_api.cu", "flce_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# (library, extra nvcc flags)
TARGETS = [(LIB, []), (DEBUG_LIB, ["-DFLCE_DEBUG"])]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflce")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "flce.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    todo = [(lib, flags) for lib, flags in TARGETS if force or not up_to_date(lib)]
    if not todo:
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(OBJDIR, exist_ok=True)
    tag = os.getpid()
    procs, objs = [], {}
    for lib, flags in todo:
        stem = os.path.splitext(os.path.basename(lib))[0]
        for src in SOURCES:
            obj = os.path.join(OBJDIR, f"{stem}.{os.path.splitext(src)[0]}.{tag}.o")
            cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   *flags, "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((f"{stem}:{src}", subprocess.Popen(
                cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
            objs.setdefault(lib, []).append(obj)
    failed = False
    for name, p in procs:
        out, err = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out)
            sys.stderr.write(err)
        if p.returncode != 0:
            print(f"nvcc failed on {name} (exit {p.returncode})", file=sys.stderr)
            failed = True
    try:
        if failed:
            raise RuntimeError("nvcc compilation failed")
        for lib, _ in todo:
            tmp = lib + f".tmp{tag}"
            link = [nvcc(), *ARCH, "-shared", "-o", tmp] + objs[lib]
            r = subprocess.run(link, capture_output=True, text=True)
            if verbose or r.returncode != 0:
                sys.stdout.write(r.stdout)
                sys.stderr.write(r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc link of {os.path.basename(lib)} failed "
                                   f"(exit {r.returncode})")
            os.replace(tmp, lib)
    finally:
        for lst in objs.values():
            for o in lst:
                try:
                    os.remove(o)
                except OSError:
                    pass
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
          ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)
    print(DEBUG_LIB)
