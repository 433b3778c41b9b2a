"""Host-side checks of the C interface that need no GPU: the library builds
for sm_103a, loads, exports every function include/mxgemm.h declares, and
rejects bad arguments without touching a device."""
import ctypes
import re
from pathlib import Path

import pytest

import block_scaled_gemm_gb300 as mx
from block_scaled_gemm_gb300 import _build

HEADER = Path(__file__).resolve().parents[1] / "include"


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mx.library()


def _declared_functions():
    names = set()
    for hdr in HEADER.glob("*.h"):
        text = hdr.read_text()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_interface():
    names = _declared_functions()
    for n in ("mxgemm_create", "mxgemm_run", "mxgemm_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    for name in mx.EXPORTED_SYMBOLS:
        assert name in _declared_functions()


def test_null_handle_rejected(lib):
    assert lib.mxgemm_run(None, 1, 1, 32, None, None, None, None, None, 0, 0, None) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_destroy(None) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_set_option(None, 1, 0) == mx.ERR_INVALID_VALUE
    st = ctypes.c_int()
    assert lib.mxgemm_get_device_status(None, None, ctypes.byref(st), None) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_create(None, 0) == mx.ERR_INVALID_VALUE


def test_status_strings(lib):
    for s in range(8):
        assert mx.mxgemm_status_string(s)
    assert "timed out" in mx.mxgemm_status_string(mx.ERR_TIMEOUT)


def test_create_without_supported_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.mxgemm_create(ctypes.byref(h), 0)
    assert st in (mx.ERR_CUDA, mx.ERR_INVALID_VALUE, mx.ERR_UNSUPPORTED_DEVICE)
    assert not h.value


def test_product_path_does_not_import_the_oracle():
    # the binding must never reach the CPU checker
    src = (Path(mx.__file__).parent).rglob("*.py")
    for f in src:
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mxgemm.h"

int main(void) {
  /* plain C: the header compiles as C, the library links and answers */
  if (strcmp(mxgemm_status_string(MXGEMM_OK), "ok") != 0) return 1;
  if (mxgemm_run(NULL, 1, 1, 32, NULL, NULL, NULL, NULL, NULL, 0, MXGEMM_OUT_F32, NULL) !=
      MXGEMM_ERR_INVALID_VALUE) return 2;
  if (mxgemm_set_option(NULL, MXGEMM_OPT_A_FORMAT, MXGEMM_FMT_E2M1) != MXGEMM_ERR_INVALID_VALUE) return 3;
  if (mxgemm_quantize(NULL, MXGEMM_IN_F32, 4, 48, 0, NULL, NULL, NULL) != MXGEMM_ERR_INVALID_VALUE)
    return 4;
  /* without a GPU: create fails cleanly, no handle */
  mxgemm_handle_t h = (mxgemm_handle_t)1;
  int st = mxgemm_create(&h, 0);
  if (st == MXGEMM_OK) { mxgemm_destroy(h); printf("gpu\n"); return 0; }
  if (h != NULL) return 5;
  printf("nogpu %d\n", st);
  return 0;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "abi_check.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi_check"
    so = mx.library_path()
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", str(HEADER), str(src), "-o", str(exe),
                        str(so), f"-Wl,-rpath,{so.parent}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.split()[0] in ("gpu", "nogpu")


def test_scale_bytes_host_only():
    # sizes of the scales in either layout, worked by hand from the layout
    # definition in mxgemm.h (no device involved)
    import block_scaled_gemm_gb300 as mx
    lib = mx.library()
    cases = [
        # R, C, along_cols, layout, bytes
        (300, 416, 0, 0, 300 * 13),               # A row-major: M x K/32
        (300, 416, 0, 1, 3 * 4 * 512),            # ceil(300/128)=3 blocks, ceil(416/128)=4 steps
        (416, 300, 1, 0, 300 * 13),               # B row-major: N x K/32
        (416, 300, 1, 1, 2 * 4 * 1024),           # ceil(300/256)=2 tiles, 4 steps
        (4096, 4096, 1, 1, 16 * 32 * 1024),
        (1, 32, 0, 1, 1 * 1 * 512),
    ]
    for R, C, ac, lay, want in cases:
        assert mx.mxgemm_scale_bytes(R, C, ac, lay) == want, (R, C, ac, lay)
    out = ctypes.c_int64(0)
    assert lib.mxgemm_scale_bytes(16, 32, 0, 2, ctypes.byref(out)) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_scale_bytes(16, 32, 0, 0, None) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_scale_bytes(16, 48, 0, 0, ctypes.byref(out)) == mx.ERR_INVALID_VALUE  # C % 32
    assert lib.mxgemm_scale_bytes(48, 16, 1, 1, ctypes.byref(out)) == mx.ERR_INVALID_VALUE  # R % 32
