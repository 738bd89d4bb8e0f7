"""In-tree build of libfa_gb300.so with nvcc for sm_103a (no CMake, no setuptools).

The translation units are compiled in parallel, then linked into a shared
library next to this file. ``build()`` is a no-op when the library is newer than
every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa_gb300.so")
LIB_TRACE = os.path.join(PKG, "libfa_gb300_trace.so")   # -DFA_TRACE: clock stamps at pipeline hand-offs
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{INCLUDE}", f"-I{CSRC}"]
UNITS = ["fa_api.cu", "fa_bwd_api.cu", "fa_selftest.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def _sources():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    lib = LIB_TRACE if trace else LIB
    if not force and up_to_date(lib):
        return lib
    exe = nvcc()
    out_dir = os.path.join(PKG, "_build")
    os.makedirs(out_dir, exist_ok=True)

    def compile_one(unit):
        obj = os.path.join(out_dir, unit.replace(".cu", f".{'t' if trace else 'n'}{os.getpid()}.o"))
        cmd = [exe, *ARCH, *FLAGS, *(["-DFA_TRACE"] if trace else []), "-c", os.path.join(CSRC, unit), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {unit}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_one, UNITS))
    objs = [o for o, _ in results]
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([exe, *ARCH, "-shared", *objs, "-o", tmp], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        for _, log in results:
            print(log)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
