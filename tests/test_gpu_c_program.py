"""The C interface used from a plain C program (no Python, no torch): device
buffers from the CUDA runtime, small-integer E4M3 operands with unit scales
(so every product and FP32 partial sum is exact), one mxgemm_run, and an exact
integer check on the host."""
import shutil
import subprocess
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_gemm_gb300")
ROOT = Path(__file__).resolve().parents[1]

C_PROGRAM = r"""
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include "mxgemm.h"

/* E4M3 codes of the integers 0..8 (1.m x 2^(E-7)); bit 7 is the sign */
static const unsigned char kCode[9] = {0x00, 0x38, 0x40, 0x44, 0x48, 0x4A, 0x4C, 0x4E, 0x50};
static unsigned char enc(int v) { return v < 0 ? (unsigned char)(0x80 | kCode[-v]) : kCode[v]; }

int main(void) {
  const int M = 300, N = 520, K = 1024;
  unsigned char *hA = malloc((size_t)M * K), *hB = malloc((size_t)K * N);
  unsigned char *hAs = malloc((size_t)M * K / 32), *hBs = malloc((size_t)N * K / 32);
  int *ia = malloc(sizeof(int) * M * K), *ib = malloc(sizeof(int) * K * N);
  float *hC = malloc(sizeof(float) * M * N);
  unsigned s = 12345;
  for (int i = 0; i < M * K; ++i) { s = s * 1103515245u + 12345u; ia[i] = (int)((s >> 16) % 17) - 8; hA[i] = enc(ia[i]); }
  for (int i = 0; i < K * N; ++i) { s = s * 1103515245u + 12345u; ib[i] = (int)((s >> 16) % 17) - 8; hB[i] = enc(ib[i]); }
  for (int i = 0; i < M * K / 32; ++i) hAs[i] = 127;
  for (int i = 0; i < N * K / 32; ++i) hBs[i] = 127;
  void *A, *As, *B, *Bs, *C;
  if (cudaMalloc(&A, (size_t)M * K) || cudaMalloc(&B, (size_t)K * N) || cudaMalloc(&As, (size_t)M * K / 32) ||
      cudaMalloc(&Bs, (size_t)N * K / 32) || cudaMalloc(&C, sizeof(float) * M * N)) return 10;
  cudaMemcpy(A, hA, (size_t)M * K, cudaMemcpyHostToDevice);
  cudaMemcpy(B, hB, (size_t)K * N, cudaMemcpyHostToDevice);
  cudaMemcpy(As, hAs, (size_t)M * K / 32, cudaMemcpyHostToDevice);
  cudaMemcpy(Bs, hBs, (size_t)N * K / 32, cudaMemcpyHostToDevice);
  mxgemm_handle_t h;
  int st = mxgemm_create(&h, 0);
  if (st) { printf("create %s\n", mxgemm_status_string(st)); return 11; }
  st = mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, MXGEMM_OUT_F32, NULL);
  if (st) { printf("run %s\n", mxgemm_status_string(st)); return 12; }
  int dst = 0, det = 0;
  if (mxgemm_get_device_status(h, NULL, &dst, &det) || dst) return 13;
  cudaMemcpy(hC, C, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
  long bad = 0;
  for (int i = 0; i < M; ++i)
    for (int j = 0; j < N; ++j) {
      long acc = 0;
      for (int k = 0; k < K; ++k) acc += (long)ia[i * K + k] * ib[k * N + j];
      if ((float)acc != hC[i * N + j]) ++bad;
    }
  mxgemm_destroy(h);
  printf("mismatches %ld\n", bad);
  return bad ? 14 : 0;
}
"""


def test_c_program_exact_integers(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    cuda = Path("/usr/local/cuda")
    src = tmp_path / "gemm.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "gemm"
    so = mx.library_path()
    r = subprocess.run([gcc, "-std=c99", "-O2", "-Wall", "-I", str(ROOT / "include"), "-I", str(cuda / "include"),
                        str(src), "-o", str(exe), str(so), f"-L{cuda / 'lib64'}", "-lcudart",
                        f"-Wl,-rpath,{so.parent}", f"-Wl,-rpath,{cuda / 'lib64'}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "mismatches 0" in r.stdout
