"""Builds libmk.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmk.so")
SOURCES = [os.path.join(CSRC, f) for f in ("mk_host.cu", "mk_kernel_dense.cu", "mk_kernel_full.cu")]
HEADERS = [os.path.join(CSRC, "mk_internal.h"), os.path.join(CSRC, "mk_kernel.cuh"), os.path.join(INCLUDE, "mk.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
    "-shared", "-Xcompiler", "-fPIC", "-I" + INCLUDE,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if a source is newer than it (or ``force``). Returns its path."""
    if not force and not stale():
        return LIB
    tmp = LIB + ".tmp"
    # the translation units compile in parallel (the two kernel builds dominate), then link
    objs = [LIB + "." + os.path.splitext(os.path.basename(src))[0] + ".o" for src in SOURCES]
    compile_flags = [f for f in NVCC_FLAGS if f != "-shared"]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [_nvcc(), *compile_flags, "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate() for p in procs]
    for p, (o, e) in zip(procs, outs):
        if p.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + o + e)
        if verbose:
            print(o + e)
    res = subprocess.run([_nvcc(), *NVCC_FLAGS, "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    for obj in objs:
        os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
    print(LIB)
