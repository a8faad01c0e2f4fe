"""Build libeng.so (the C-ABI library of include/eng.h) in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into
graph_replayed_decode_gb300/libeng.so.  The units whose kernels depend on the 16-bit element format
(ELEMENT_UNITS) are compiled a second time with ENG_F16 defined, for the fp16 variant of a model (their
symbols then live in the namespace grd::f16; see csrc/common.cuh).
Usage: ``python -m graph_replayed_decode_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libeng.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing",
              "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: libeng.so cannot be built")
    return path


ELEMENT_UNITS = ("gemm.cu", "attn_decode.cu", "attn_prefill.cu", "norm.cu", "pack.cu")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def units() -> list[tuple[str, bool]]:
    """(source, fp16 build) of every object: each source once, the element-format units twice."""
    return [(s, False) for s in sources()] + [(s, True) for s in sources() if os.path.basename(s) in ELEMENT_UNITS]


def _compile(unit: tuple[str, bool], extra: list[str]) -> tuple[str, str]:
    src, f16 = unit
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ("_f16.o" if f16 else ".o"))
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, *(["-DENG_F16"] if f16 else []), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    us = units()
    with cf.ThreadPoolExecutor(max_workers=min(len(us), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda u: _compile(u, extra), us))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
