"""Build libditsp.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into sequence_attention_gb300/libditsp.so with a static
CUDA runtime, so the library needs only the driver at run time.

    python sequence_attention_gb300/build.py [-v] [--ptxas]

(run as a script: importing the package needs the library this produces)
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libditsp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden",
          f"-I{INCLUDE}", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libditsp")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"command failed ({p.returncode}): {' '.join(cmd)}\n{p.stdout}")
    if verbose and p.stdout.strip():
        print(p.stdout, flush=True)
    return p.stdout


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    srcs = sources()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(pair):
        src, obj = pair
        return _run([cc, *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj], verbose or ptxas_info)

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        outs = list(ex.map(compile_one, zip(srcs, objs)))
    if ptxas_info:
        for o in outs:
            sys.stdout.write(o)
    tmp = LIB + ".tmp"
    _run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], verbose)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose=v, ptxas_info="--ptxas" in sys.argv))
