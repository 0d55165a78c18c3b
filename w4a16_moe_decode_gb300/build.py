"""Builds libflint_moe.so in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel, then one shared library is
linked against the CUDA runtime. No CMake, no torch extension machinery: the
library exposes a plain C ABI (include/flint_moe.h, include/flint_synth.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.environ.get("FLINT_MOE_LIB") or os.path.join(PKG, "libflint_moe.so")
SOURCES = ["decode.cu", "pack.cu", "synth.cu", "prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflint_moe.so")


def _compile(src: str, verbose_ptxas: bool, defines=()) -> str:
    suffix = ("_" + "_".join(d.lower() for d in defines)) if defines else ""
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + suffix + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
           "-I", INCLUDE, "-I", CSRC, *("-D" + d for d in defines), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        print(res.stderr)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
           [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, trace: bool = False, out: str | None = None) -> str:
    """Compiles the library if a source is newer than it; returns its path.
    trace=True builds the phase-trace variant (flint_moe_trace records) into
    `out` (default libflint_moe_trace.so beside the normal library)."""
    lib = out or (os.path.join(PKG, "libflint_moe_trace.so") if trace else LIB)
    if not force and not trace and not _stale():
        return lib
    os.makedirs(BUILD, exist_ok=True)
    defines = ("FLINT_MOE_TRACE",) if trace else ()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, defines), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
