"""Build the sm_103a shared library ``libcsa_b300.so`` in-tree with nvcc.

Every kernel is compiled for ``-gencode arch=compute_103a,code=sm_103a`` only;
the library links the CUDA runtime statically and resolves the driver's
tensor-map encoder at run time, so no libcuda link is needed at build time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcsa_b300.so")
SOURCES = ["api.cu", "compress.cu", "indexer.cu", "topk.cu", "topk_noalloc.cu", "attn.cu", "attn_tc.cu", "decode.cu"]
HEADERS = ["common.cuh", "kernels.h"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr", "-rdc=true",
    "-Xptxas", "-warn-spills",
    "-I", os.path.join(ROOT, "include"),
]


def _newest_dep() -> float:
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "csa.h"),
                                                       os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in deps)


def _compile(src: str, force: bool, verbose_ptxas: bool) -> str:
    obj = os.path.join(OBJ, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), _newest_dep()):
        return obj
    cmd = [NVCC, *FLAGS, "-c", path, "-o", obj]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.check_call(cmd)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force, verbose_ptxas), SOURCES))
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-rdc=true", "-shared", *objs,
                               "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
