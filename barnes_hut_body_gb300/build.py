"""Compile libbh.so in-tree for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel, then linked with nvcc into
``barnes_hut_body_gb300/libbh.so``.  Objects go to ``barnes_hut_body_gb300/_build``.

    python -m barnes_hut_body_gb300.build [-v] [--ptxas-v]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbh.so")
SOURCES = ["bh_api.cu", "k_keys_sort.cu", "k_build.cu", "k_walk.cu", "k_direct.cu",
           "k_integrate.cu", "k_sbh.cu", "k_nbr.cu", "k_order.cu", "k_peak.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_v: bool) -> list[str]:
    f = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
         "-I", INCLUDE, "-I", CSRC]
    if ptxas_v:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose: bool = False, ptxas_v: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    cc = nvcc()
    flags = _flags(ptxas_v)

    def one(src: str) -> str:
        out = os.path.join(OBJ, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", out]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if (verbose or ptxas_v) and r.stderr:
            print(r.stderr, file=sys.stderr, flush=True)
        return out

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_v="--ptxas-v" in sys.argv))
