"""Build libfi_nvfp4.so (and the diagnostic probe library) in-tree with nvcc.

    python nvfp4_paged_kv_slot_b300/build.py [--force] [-v]

The script uses the standard library only, so it runs before the package (whose
import needs the built library) can be imported.

Targets sm_103a only.  No fast-math: the quantizer relies on IEEE division
and separately rounded products (it uses explicit _rn intrinsics as well).
"""
from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import sys

HERE = pathlib.Path(__file__).resolve().parent
ROOT = HERE.parent
CSRC = HERE / "csrc"
INCLUDE = ROOT / "include"
LIB = HERE / "libfi_nvfp4.so"
DIAG_LIB = HERE / "libfi_nvfp4_diag.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]

LIB_SOURCES = ["api.cu", "append.cu", "prefill.cu", "decode.cu", "planner.cpp", "noalloc.cu"]
DIAG_SOURCES = ["diag.cu"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return p


def _stale(target: pathlib.Path, sources) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    deps = list(sources) + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        list(INCLUDE.glob("*.h")) + [pathlib.Path(__file__)]
    return any(d.stat().st_mtime > t for d in deps)


def _compile(target: pathlib.Path, sources, extra=(), verbose=False):
    tmp = target.with_suffix(f".so.tmp{os.getpid()}")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-I", str(INCLUDE), "-I", str(CSRC),
           *[str(s) for s in sources], "-o", str(tmp)]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)


def build(force: bool = False, verbose: bool = False) -> pathlib.Path:
    srcs = [CSRC / s for s in LIB_SOURCES]
    if force or _stale(LIB, srcs):
        _compile(LIB, srcs, verbose=verbose)
    dsrcs = [CSRC / s for s in DIAG_SOURCES]
    if force or _stale(DIAG_LIB, dsrcs):
        _compile(DIAG_LIB, dsrcs, verbose=verbose)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
