"""Builds the gbtopk shared library in-tree for sm_103a with nvcc.

The two translation units are compiled in parallel and linked into
``sparse_attention_top_gb300/libgbtopk.so`` (CUDA runtime linked statically).
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
LIB = os.path.join(PKG, "libgbtopk.so")
SOURCES = ["gbtopk_api.cu", "gbtopk_kernels.cu", "gbtopk_static_ws.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the gbtopk CUDA library cannot be built")
    return cand


def _compile(src: str, obj: str, extra) -> None:
    cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj, *extra]
    subprocess.check_call(cmd)


def build(verbose_ptxas: bool = False) -> str:
    """Compile and link; returns the library path."""
    bdir = os.path.join(PKG, "_build")
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        list(ex.map(lambda a: _compile(a[0], a[1], extra), zip(SOURCES, objs)))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
