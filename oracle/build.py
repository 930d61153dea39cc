"""Compile the CPU oracle (oracle.cpp) into oracle/liboracle.so with g++.

Test infrastructure: the product library never links or loads this.
"""
import os
import pathlib
import subprocess
import sys

HERE = pathlib.Path(__file__).resolve().parent
SRC = HERE / "oracle.cpp"
HDR = HERE / "oracle.h"
LIB = HERE / "liboracle.so"

# -ffp-contract=off: every fp32 step of the quantizer stays a separately rounded
# IEEE operation (no fused multiply-add), which is what the oracle specifies.
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
         "-fno-fast-math", "-Wall", "-Wextra"]


def needs_build() -> bool:
    if not LIB.exists():
        return True
    lib_t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > lib_t for p in (SRC, HDR, pathlib.Path(__file__)))


def build(force: bool = False) -> pathlib.Path:
    if force or needs_build():
        tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["g++", *FLAGS, str(SRC), "-o", str(tmp)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
