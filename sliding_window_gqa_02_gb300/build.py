"""Build ``libgqaw.so`` (the C-ABI library of include/gqaw.h) in-tree with nvcc.

The CUDA sources are compiled for sm_103a only, one object per translation unit, in
parallel, then linked into ``sliding_window_gqa_02_gb300/_lib/libgqaw.so``.  Objects
are rebuilt when their source or any header is newer.
"""
from __future__ import annotations

import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libgqaw.so")

SOURCES = ["gqaw_host.cu", "gqaw_finish.cu", "gqaw_attend_f32.cu", "gqaw_attend_bf16.cu", "gqaw_noalloc.cu", "gqaw_mma.cu",
           "gqaw_rotary.cu", "gqaw_mmad.cu", "gqaw_attend_q8.cu", "gqaw_quant.cu",
           "gqaw_mmad_q8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _headers_mtime():
    paths = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, hdr_mtime: float) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), hdr_mtime):
        return obj
    log = os.path.join(BUILD, os.path.splitext(src)[0] + ".ptxas.log")
    cmd = [_nvcc(), *ARCH, *FLAGS, "-c", path, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stderr[-6000:]))
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False) -> str:
    """Compile and link libgqaw.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    # Objects built on another host architecture (x86_64 vs aarch64) are never reused.
    stamp = os.path.join(BUILD, "host.txt")
    host = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != host:
        force = True
    if force:
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
    hdr = _headers_mtime()
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, hdr), SOURCES))
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s" % r.stderr[-6000:])
        os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(host + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
