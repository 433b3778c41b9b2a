"""Build step for the CUDA library: sm_103a only, one nvcc compile per
translation unit (run in parallel), then one link.

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
# translation units: the C interface with the tiled kernel (B given K x N),
# the tiled kernel's variants for B given N x K, and the skinny-problem kernel
UNITS = [SRC_DIR / "mxgemm.cu", SRC_DIR / "tiled_kmajor.cu", SRC_DIR / "swapab.cu"]
OBJ_DIR = PKG / "_build"
HEADER = ROOT / "include" / "mxgemm.h"
LIB = PKG / "libmxgemm.so"

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-std=c++17", "-O3", "-lineinfo",
    "-Xcompiler", "-fPIC",
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
    nvcc = nvcc_path()
    OBJ_DIR.mkdir(exist_ok=True)
    tag = os.getpid()
    objs, procs = [], []
    for src in UNITS:
        obj = OBJ_DIR / f"{src.stem}.{tag}.o"
        cmd = [nvcc, *NVCC_FLAGS, "-I", str(ROOT / "include"), "-c", "-o", str(obj), str(src)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), file=sys.stderr)
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, pr in procs if pr.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    tmp = LIB.with_name(f"libmxgemm.so.tmp{tag}")
    subprocess.run([nvcc, "-shared", "-Xcompiler", "-fPIC", "-o", str(tmp), *map(str, objs)],
                   check=True)
    for obj in objs:
        obj.unlink()
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
