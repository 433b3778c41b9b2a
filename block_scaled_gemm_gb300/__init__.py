"""Python binding of the GB300 MX block-scaled FP8 GEMM C library.

Argument marshalling only: every step of the product runs in the CUDA
library ``libmxgemm.so`` (built from ``csrc/`` by ``_build.build()``); there is
no fallback.  The functions mirror the C interface of ``include/mxgemm.h``:

    h = mxgemm_create(device)
    mxgemm_run(h, M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, stream)
    mxgemm_destroy(h)

Tensor arguments may be anything with ``data_ptr()`` (torch CUDA tensors) or
raw integer device addresses.  ``stream`` may be a ``torch.cuda.Stream``, a
raw ``cudaStream_t`` integer, or None (the legacy default stream).
The operation is the scaled product documented as ``tlx.async_dot_scaled``
("TLX API Quick Reference", section "Matrix Multiply (MMA)").
"""
from __future__ import annotations

import ctypes
from pathlib import Path

from . import _build

__all__ = [
    "OUT_F32", "OUT_BF16", "OPT_MODE", "OPT_WAIT_TIMEOUT_NS", "OPT_TEST_STALL_PRODUCER",
    "OPT_SCHEDULER", "OPT_STREAM_K", "OPT_A_FORMAT", "OPT_B_FORMAT", "FMT_E4M3", "FMT_E5M2",
    "FMT_E2M3", "FMT_E3M2", "FMT_E2M1", "MxgemmError", "library", "library_path", "mxgemm_create", "mxgemm_run",
    "mxgemm_destroy", "mxgemm_set_option", "mxgemm_get_device_status", "mxgemm_status_string",
    "mxgemm_set_profile_events", "mxgemm_get_launch_count", "mxgemm_run_noalloc", "mxgemm_run_host",
    "mxgemm_quantize", "IN_F32", "IN_BF16", "EXPORTED_SYMBOLS", "Gemm", "OPT_SCALE_LAYOUT", "OPT_ELEMENT_LAYOUT", "OPT_B_MAJOR", "B_K_BY_N", "B_N_BY_K", "ELEMS_BYTE", "ELEMS_PACKED",
    "SCALES_ROW_MAJOR", "SCALES_PACKED", "mxgemm_scale_bytes", "mxgemm_noalloc_get_status",
    "mxgemm_noalloc_set_option",
]

OUT_F32 = 0
OUT_BF16 = 1

OPT_MODE = 1
OPT_WAIT_TIMEOUT_NS = 2
OPT_TEST_STALL_PRODUCER = 3
OPT_SCHEDULER = 4
OPT_STREAM_K = 5
OPT_A_FORMAT = 6
OPT_B_FORMAT = 7
OPT_SCALE_LAYOUT = 8
OPT_ELEMENT_LAYOUT = 10
OPT_B_MAJOR = 11
B_K_BY_N = 0
B_N_BY_K = 1
ELEMS_BYTE = 0
ELEMS_PACKED = 1

# scale layouts (mxgemm_scale_layout_t)
SCALES_ROW_MAJOR = 0
SCALES_PACKED = 1

# element formats (mxgemm_format_t); one element per byte, sub-byte codes in
# the low bits
FMT_E4M3 = 0
FMT_E5M2 = 1
FMT_E2M3 = 2
FMT_E3M2 = 3
FMT_E2M1 = 4

OK = 0
ERR_INVALID_VALUE = 1
ERR_MISALIGNED = 2
ERR_UNSUPPORTED_DEVICE = 3
ERR_OUT_OF_MEMORY = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
ERR_TOO_LARGE = 7

EXPORTED_SYMBOLS = (
    "mxgemm_create", "mxgemm_run", "mxgemm_destroy", "mxgemm_set_option",
    "mxgemm_get_device_status", "mxgemm_status_string", "mxgemm_set_profile_events",
    "mxgemm_get_launch_count", "mxgemm_run_noalloc", "mxgemm_run_host", "mxgemm_quantize",
    "mxgemm_quantize_sr", "mxgemm_quantize_ex", "mxgemm_scale_bytes", "mxgemm_noalloc_get_status",
    "mxgemm_noalloc_set_option",
)

_lib = None


class MxgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mxgemm_status_string(status)} (status {status})")


def library_path() -> Path:
    return _build.LIB


def library():
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not path.exists():
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with "
                "`python -m block_scaled_gemm_gb300._build` (there is no CPU fallback)")
        lib = ctypes.CDLL(str(path))
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.mxgemm_create.argtypes = [ctypes.POINTER(vp), i32]
        lib.mxgemm_create.restype = i32
        lib.mxgemm_run.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, i32, vp]
        lib.mxgemm_run.restype = i32
        lib.mxgemm_destroy.argtypes = [vp]
        lib.mxgemm_destroy.restype = i32
        lib.mxgemm_set_option.argtypes = [vp, i32, i64]
        lib.mxgemm_set_option.restype = i32
        lib.mxgemm_get_device_status.argtypes = [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.mxgemm_get_device_status.restype = i32
        lib.mxgemm_set_profile_events.argtypes = [vp, vp, vp]
        lib.mxgemm_set_profile_events.restype = i32
        lib.mxgemm_get_launch_count.argtypes = [vp, ctypes.POINTER(i64)]
        lib.mxgemm_get_launch_count.restype = i32
        lib.mxgemm_quantize.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp]
        lib.mxgemm_quantize.restype = i32
        lib.mxgemm_quantize_sr.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp, vp]
        lib.mxgemm_quantize_sr.restype = i32
        lib.mxgemm_quantize_ex.argtypes = [vp, i32, i64, i64, i32, vp, i32, vp, vp, vp]
        lib.mxgemm_quantize_ex.restype = i32
        lib.mxgemm_scale_bytes.argtypes = [i64, i64, i32, i32, ctypes.POINTER(i64)]
        lib.mxgemm_scale_bytes.restype = i32
        lib.mxgemm_run_host.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, i32, vp]
        lib.mxgemm_run_host.restype = i32
        lib.mxgemm_run_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, i32, i32, vp]
        lib.mxgemm_run_noalloc.restype = i32
        lib.mxgemm_noalloc_get_status.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.mxgemm_noalloc_get_status.restype = i32
        lib.mxgemm_noalloc_set_option.argtypes = [i32, i64]
        lib.mxgemm_noalloc_set_option.restype = i32
        lib.mxgemm_status_string.argtypes = [i32]
        lib.mxgemm_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def mxgemm_status_string(status: int) -> str:
    return library().mxgemm_status_string(int(status)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != OK:
        raise MxgemmError(st, where)


def mxgemm_create(device: int = 0):
    h = ctypes.c_void_p()
    _check(library().mxgemm_create(ctypes.byref(h), int(device)), "mxgemm_create")
    return h


def mxgemm_run(h, M, N, K, A, A_scale, B, B_scale, C, use_acc=0, out_dtype=OUT_F32, stream=None,
               check: bool = True) -> int:
    st = library().mxgemm_run(h, int(M), int(N), int(K), _ptr(A), _ptr(A_scale), _ptr(B),
                              _ptr(B_scale), _ptr(C), int(bool(use_acc)), int(out_dtype),
                              _stream(stream))
    if check:
        _check(st, "mxgemm_run")
    return st


IN_F32 = 0
IN_BF16 = 1


def mxgemm_quantize(X, R, C, codes, scales, along_cols=False, x_dtype=None, stream=None,
                    check: bool = True, rand_bits=None, scale_layout=SCALES_ROW_MAJOR) -> int:
    """MX-quantize the R x C device matrix X (float32 or bfloat16) into E4M3
    codes (R x C bytes) and E8M0 scales per 32 values, along the rows
    (A_scale of an M x K X) or down the columns (B_scale of a K x N X).
    With rand_bits (an R x C device tensor of 32-bit words) the codes round
    stochastically, else to nearest even.  scale_layout SCALES_ROW_MAJOR
    gives R x C/32 (rows) or C x R/32 (columns) scales, SCALES_PACKED the
    order a run with OPT_SCALE_LAYOUT = SCALES_PACKED reads
    (mxgemm_scale_bytes bytes)."""
    if x_dtype is None:
        import torch
        x_dtype = IN_BF16 if getattr(X, "dtype", None) == torch.bfloat16 else IN_F32
    lib = library()
    if rand_bits is None and scale_layout == SCALES_ROW_MAJOR:
        st = lib.mxgemm_quantize(_ptr(X), int(x_dtype), int(R), int(C), int(bool(along_cols)),
                                 _ptr(codes), _ptr(scales), _stream(stream))
        name = "mxgemm_quantize"
    elif scale_layout == SCALES_ROW_MAJOR:
        st = lib.mxgemm_quantize_sr(_ptr(X), int(x_dtype), int(R), int(C), int(bool(along_cols)),
                                    _ptr(rand_bits), _ptr(codes), _ptr(scales), _stream(stream))
        name = "mxgemm_quantize_sr"
    else:
        st = lib.mxgemm_quantize_ex(_ptr(X), int(x_dtype), int(R), int(C), int(bool(along_cols)),
                                    _ptr(rand_bits), int(scale_layout), _ptr(codes), _ptr(scales),
                                    _stream(stream))
        name = "mxgemm_quantize_ex"
    if check:
        _check(st, name)
    return st


def mxgemm_scale_bytes(R, C, along_cols=False, scale_layout=SCALES_ROW_MAJOR) -> int:
    """Bytes of the scales of an R x C matrix quantized along the rows or
    down the columns, in the given layout."""
    out = ctypes.c_int64(0)
    _check(library().mxgemm_scale_bytes(int(R), int(C), int(bool(along_cols)), int(scale_layout),
                                        ctypes.byref(out)), "mxgemm_scale_bytes")
    return int(out.value)


def mxgemm_run_host(h, M, N, K, A, A_scale, B, B_scale, C, use_acc=0, out_dtype=OUT_F32,
                    stream=None, check: bool = True) -> int:
    """C (+)= A.B with every operand and C in host memory (CPU tensors,
    contiguous; pinned ones let the copies overlap the GEMM).  C is complete
    once `stream` is synchronized (see include/mxgemm.h)."""
    st = library().mxgemm_run_host(h, int(M), int(N), int(K), _ptr(A), _ptr(A_scale), _ptr(B),
                                   _ptr(B_scale), _ptr(C), int(bool(use_acc)), int(out_dtype),
                                   _stream(stream))
    if check:
        _check(st, "mxgemm_run_host")
    return st


def mxgemm_run_noalloc(M, N, K, A, A_scale, B, B_scale, C, use_acc=0, out_dtype=OUT_F32,
                       stream=None, check: bool = True) -> int:
    """C (+)= A.B on the current device without allocating device memory
    (fixed 16 MiB scratch shared by all calls; see include/mxgemm.h)."""
    st = library().mxgemm_run_noalloc(int(M), int(N), int(K), _ptr(A), _ptr(A_scale), _ptr(B),
                                      _ptr(B_scale), _ptr(C), int(bool(use_acc)), int(out_dtype),
                                      _stream(stream))
    if check:
        _check(st, "mxgemm_run_noalloc")
    return st


def mxgemm_noalloc_get_status(stream=None):
    """Synchronize `stream`, then read and clear the current device's status
    word of mxgemm_run_noalloc: (status, detail), the first failure since the
    last read."""
    st, det = ctypes.c_int(), ctypes.c_int()
    _check(library().mxgemm_noalloc_get_status(_stream(stream), ctypes.byref(st), ctypes.byref(det)),
           "mxgemm_noalloc_get_status")
    return st.value, det.value


def mxgemm_noalloc_set_option(option: int, value: int) -> None:
    """Process-wide option of mxgemm_run_noalloc (OPT_WAIT_TIMEOUT_NS or
    OPT_TEST_STALL_PRODUCER)."""
    _check(library().mxgemm_noalloc_set_option(int(option), int(value)), "mxgemm_noalloc_set_option")


def mxgemm_set_option(h, option: int, value: int) -> None:
    _check(library().mxgemm_set_option(h, int(option), int(value)), "mxgemm_set_option")


def mxgemm_get_device_status(h, stream=None):
    st, det = ctypes.c_int(), ctypes.c_int()
    _check(library().mxgemm_get_device_status(h, _stream(stream), ctypes.byref(st), ctypes.byref(det)),
           "mxgemm_get_device_status")
    return st.value, det.value


def mxgemm_set_profile_events(h, ev_before, ev_after) -> None:
    """Record these CUDA events (torch.cuda.Event, raw handles or None)
    around the GEMM kernel launch of later runs.  torch events must already
    have been recorded once (torch creates the CUDA event lazily)."""
    def raw(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    _check(library().mxgemm_set_profile_events(h, raw(ev_before), raw(ev_after)),
           "mxgemm_set_profile_events")


def mxgemm_get_launch_count(h) -> int:
    n = ctypes.c_int64()
    _check(library().mxgemm_get_launch_count(h, ctypes.byref(n)), "mxgemm_get_launch_count")
    return n.value


def mxgemm_destroy(h) -> None:
    _check(library().mxgemm_destroy(h), "mxgemm_destroy")


class Gemm:
    """Owns one handle.  ``g(A, As, B, Bs, C, use_acc, out_dtype)`` enqueues
    C (+)= A.B on the current torch stream (shapes taken from the tensors)."""

    def __init__(self, device: int = 0, mode: int | None = None):
        self.h = mxgemm_create(device)
        if mode is not None:
            mxgemm_set_option(self.h, OPT_MODE, mode)

    def __call__(self, A, A_scale, B, B_scale, C, use_acc=False, out_dtype=OUT_F32, stream=None):
        M, K = A.shape
        N = B.shape[1]
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(A.device)
        return mxgemm_run(self.h, M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, stream)

    def set_option(self, option: int, value: int):
        mxgemm_set_option(self.h, option, value)

    def status(self, stream=None):
        return mxgemm_get_device_status(self.h, stream)

    def close(self):
        if self.h is not None:
            mxgemm_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
