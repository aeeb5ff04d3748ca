"""Build libsmoe.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel, then one link. No cmake.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libsmoe.so")
SOURCES = ["smoe_api.cu", "route.cu", "decode.cu", "decode_stack.cu", "prefill.cu", "noalloc.cu", "cache.cu", "debug.cu",
           "deltanet.cu", "quant.cu"]
HEADERS = ["smoe_dev.cuh", "smoe_internal.h", "decode_common.cuh", "route_common.cuh"]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing", "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libsmoe.so")
    return cand


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "smoe.h")]
    if not force and not _stale(LIB, deps):
        return LIB
    bdir = os.path.join(ROOT, "_build", "smoe")
    os.makedirs(bdir, exist_ok=True)
    procs, objs = [], []
    for s in SOURCES:
        obj = os.path.join(bdir, s.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc()] + NVCC_FLAGS + ["-I", os.path.join(ROOT, "include"), "-c",
                                       os.path.join(CSRC, s), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out)
        if p.returncode:
            failed.append(s)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp] + objs,
                   check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
