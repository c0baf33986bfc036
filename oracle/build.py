"""Compile the CPU oracle (plain C, gcc + OpenMP) into oracle/_build/.

Test infrastructure only: the tests, the smoke check and the benchmark's CPU
baseline load what this builds; the CUDA library never does.  The same source is
built twice, once with fp32 arithmetic and once with fp64.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "blasst_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    objs = []
    for real, suffix in (("float", "_f32"), ("double", "_f64")):
        obj = os.path.join(OUT_DIR, f"oracle{suffix}.o")
        cmd = ["gcc", "-O2", "-fPIC", "-fopenmp", "-std=c11", "-Wall", "-Wextra",
               "-fno-fast-math", "-ffp-contract=off",
               f"-DREAL={real}", f"-DSUFFIX={suffix}", "-c", SRC, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        subprocess.run(cmd, check=True)
        objs.append(obj)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-shared", "-fopenmp", "-o", tmp, *objs, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
