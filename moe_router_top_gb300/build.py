"""Build libsmr.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the shared object links the CUDA
runtime statically and exports only the smr_* C symbols. Output:
moe_router_top_gb300/_build/libsmr.so (git-ignored).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsmr.so")
SOURCES = ["smr_api.cpp", "smr_small.cu", "smr_align.cu", "smr_tc.cu", "smr_select.cu", "smr_expert.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("smr_device.cuh", "smr_launch.h")] + [
    os.path.join(INCLUDE, "smr.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division/sqrt and no flush-to-zero: weights are compared at 2e-6
# relative and logits may be subnormal; FMA contraction stays on.
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
         "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or CUDA_HOME)")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(OUT, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + ARCH + FLAGS + (["-Xptxas", "-v"] if ptxas_verbose and src.endswith(".cu") else [])
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"--- {src} ---\n{text}")
        elif (verbose or ptxas_verbose) and text.strip():
            print(f"--- {src} ---\n{text}", file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc] + ARCH + ["-shared", "-o", tmp] + objs + [
        "-cudart", "static", "-Xlinker", "--exclude-libs,ALL", "-lrt", "-ldl", "-lpthread"]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    subprocess.check_call(link)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv))
