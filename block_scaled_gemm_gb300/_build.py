"""Build step for the CUDA library: one nvcc invocation, sm_103a only.

    python -m block_scaled_gemm_gb300._build        # (re)build libmxgemm.so

The library is built in-tree (``block_scaled_gemm_gb300/libmxgemm.so``, not
committed) so that the process that uses it loads it from the package.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SRC_DIR = PKG / "csrc"
MAIN_SRC = SRC_DIR / "mxgemm.cu"
HEADER = ROOT / "include" / "mxgemm.h"
LIB = PKG / "libmxgemm.so"

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-std=c++17", "-O3", "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda")) / "bin" / "nvcc"
    if cand.exists():
        return str(cand)
    raise RuntimeError("nvcc not found (set CUDA_HOME or put nvcc on PATH)")


def _sources():
    return [HEADER] + sorted(SRC_DIR.glob("*.cu")) + sorted(SRC_DIR.glob("*.cuh"))


def needs_build() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(s.stat().st_mtime > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not needs_build():
        return LIB
    tmp = LIB.with_name(f"libmxgemm.so.tmp{os.getpid()}")
    cmd = [nvcc_path(), *NVCC_FLAGS, "-I", str(ROOT / "include"), "-o", str(tmp), str(MAIN_SRC)]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
