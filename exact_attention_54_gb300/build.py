"""Compile the CUDA sources into the in-tree shared library libfa.so.

nvcc, sm_103a only (-gencode arch=compute_103a,code=sm_103a), one object per
translation unit compiled in parallel, static CUDA runtime. The library has no
dependency on libcuda at link time: the tensor-map encoder is fetched from the
driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
SELFTEST_LIB = os.path.join(PKG, "libfa_selftest.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"]


# library -> its translation units
TARGETS = {
    LIB: lambda: sorted(glob.glob(os.path.join(CSRC, "*.cu"))),
    SELFTEST_LIB: lambda: sorted(glob.glob(os.path.join(CSRC, "selftest", "*.cu"))),
}


def _deps(srcs):
    return sorted(set(srcs) | set(glob.glob(os.path.join(CSRC, "*.cuh"))) |
                  set(glob.glob(os.path.join(CSRC, "*.h"))) | {os.path.join(ROOT, "include", "fa.h")})


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.relpath(src, CSRC).replace(os.sep, "_") + ".o")
    cmd = [NVCC, *ARCH, *CFLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libfa.so and the test-only libfa_selftest.so when any of their
    sources is newer; returns the path of libfa.so."""
    os.makedirs(BUILD, exist_ok=True)
    todo = {lib: srcs() for lib, srcs in TARGETS.items()}
    todo = {lib: srcs for lib, srcs in todo.items() if force or verbose or _stale(lib, _deps(srcs))}
    if not todo:
        return LIB
    all_srcs = [s for srcs in todo.values() for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(all_srcs), os.cpu_count() or 1))) as ex:
        objs = dict(zip(all_srcs, ex.map(lambda s: _compile(s, verbose), all_srcs)))
    if verbose:
        for _, log in objs.values():
            sys.stderr.write(log)
    for lib, srcs in todo.items():
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *[objs[s][0] for s in srcs]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {lib} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
