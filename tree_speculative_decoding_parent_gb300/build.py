"""Build libgt.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc.

Each source compiles to an object under ``_build/`` in parallel, then nvcc links the
shared library next to this file. ``build(check=True)`` builds the checked flavour,
libgt_check.so (``-DGT_CHECK=1``: extra device-side input checks that report through the
error word), from the same sources into ``_build_check/``. Nothing is installed outside the
package directory.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgt.so")
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libgt_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(nvcc: str, src: str, verbose_ptxas: bool, check: bool = False) -> str:
    obj = os.path.join(BUILD_CHECK if check else BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, "-Xcompiler", "-fPIC,-fvisibility=hidden", "-c", src, "-o", obj]
    if check:
        cmd.insert(1, "-DGT_CHECK=1")
    if src.endswith(".cpp"):
        cmd[cmd.index("-c"):cmd.index("-c")] = ["-x", "cu"]
    if verbose_ptxas and src.endswith(".cu"):
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, check: bool = False) -> str:
    """Compile every CUDA/C++ source and link libgt.so (check: libgt_check.so); returns the
    library path."""
    lib, bdir = (LIB_CHECK, BUILD_CHECK) if check else (LIB, BUILD)
    srcs = sources()
    newest = max(os.path.getmtime(p) for p in srcs + [os.path.join(ROOT, "include", "gt.h")] +
                 [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")])
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose_ptxas, check), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                check="--check" in sys.argv))
