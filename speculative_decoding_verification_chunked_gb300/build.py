"""Builds the CUDA library ``libsvx.so`` in-tree for sm_103a, and its bounds-checked
variant ``libsvx_checked.so`` (-DSVX_BOUNDS_CHECK: every kernel checks its global
accesses against the buffers its launch describes and reports a stray one through
the device error word instead of making it).

Each translation unit is compiled by its own nvcc process (all in parallel), then
linked into one shared library next to this file.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsvx.so")
LIB_CHECKED = os.path.join(PKG, "libsvx_checked.so")

SOURCES = ["svx_kernels.cu", "svx_tc_kernel.cu", "svx_runtime.cu", "svx_static.cu", "svx_tier.cu", "svx_sched.cu", "svx_width.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xcompiler", "-ffp-contract=off",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsvx.so")


def build(verbose: bool = False, extra_flags: tuple = (), checked: bool = True) -> str:
    """Compiles every translation unit (both variants at once when `checked`) and links libsvx.so, then
    libsvx_checked.so.  Returns the path of libsvx.so."""
    cc = nvcc()
    variants = [("", LIB, ())] + ([("checked", LIB_CHECKED, ("-DSVX_BOUNDS_CHECK",))] if checked else [])
    procs, objs = [], {}
    for sub, lib, flags in variants:
        bdir = os.path.join(BUILD, sub) if sub else BUILD
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            obj = os.path.join(bdir, src.replace(".cu", ".o"))
            cmd = [cc, *ARCH, *FLAGS, *flags, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
            objs.setdefault(lib, []).append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    for _sub, lib, _flags in variants:
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs[lib]]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
