"""Build the C++ oracle (test infrastructure) with g++: a single-threaded library and the same
source with OpenMP across all host cores.

Both are built with -ffp-contract=off (no fused multiply-add), -O2 and no machine-specific
flags, so they compile and give the same results on x86-64 and Arm hosts.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gift_oracle.cpp")
LIB_SERIAL = os.path.join(HERE, "libgift_oracle.so")
LIB_OMP = os.path.join(HERE, "libgift_oracle_omp.so")
FLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wno-unknown-pragmas"]


def _cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand:
            return cand
    raise RuntimeError("no C++ compiler found to build the oracle")


def _build_one(out: str, extra) -> str:
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    r = subprocess.run([_cxx(), *FLAGS, *extra, SRC, "-o", out + ".tmp"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(out + ".tmp", out)
    return out


def build(openmp: bool = True) -> list:
    libs = [_build_one(LIB_SERIAL, [])]
    if openmp:
        libs.append(_build_one(LIB_OMP, ["-fopenmp"]))
    return libs


if __name__ == "__main__":
    for p in build():
        print(p)
