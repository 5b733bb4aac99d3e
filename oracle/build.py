"""Compile the oracle (plain C, OpenMP) to ``oracle/liborc.so``.

Test infrastructure only.  IEEE fp32 semantics are required for the bounding
cube and Morton quantisation, hence ``-ffp-contract=off`` and no fast-math.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    src = os.path.join(HERE, "bh_oracle.c")
    out = os.path.join(HERE, "liborc.so")
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
