"""Plain CPU oracle for the block-scaled (MX) matrix product.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path
(``block_scaled_gemm_gb300``) never imports it and shares no code with it.

What it computes is the plain definition of the scaled product documented as
``tlx.async_dot_scaled`` ("TLX API Quick Reference", section "Matrix Multiply
(MMA)": D = (A*scale_A) @ (B*scale_B) + D with FP8 operands), with E4M3
elements and E8M0 scales per 32 consecutive K elements (OCP Microscaling
Formats v1.0):

    ref[i, j]   = [use_acc] * C_in[i, j]
                  + sum_k e4m3(A[i,k]) e8m0(As[i,k//32]) e4m3(B[k,j]) e8m0(Bs[j,k//32])
    bound[i, j] = [use_acc] * |C_in[i, j]| + sum_k |same term|

in IEEE double, k ascending (the C file ``mxoracle.c`` does the sum).

Pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``:
decoder values against the format definitions and an independent library
decode, hand-computed tiny cases (``tests/golden/``), all-scales-127 against
a library FP64 matmul, scale-shift linearity, exact small-integer products
against an int64 matmul, exact-rational brute force on tiny inputs, and
K-split / transpose identities.  The GPU's own accumulation order is not
modelled: that part of parity is governed by the tolerance in ``accept``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "mxoracle.c"
_LIB_PATH = _HERE / "libmxoracle.so"
_lib = None

FLT_MAX = float(np.finfo(np.float32).max)


def build(force: bool = False) -> Path:
    """Compile ``mxoracle.c`` with the host's gcc into ``libmxoracle.so``."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        i64, u8p, i64p, f64p = (ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p)
        lib.mxo_e4m3.argtypes = [ctypes.c_uint8]
        lib.mxo_e4m3.restype = ctypes.c_double
        lib.mxo_e8m0.argtypes = [ctypes.c_uint8]
        lib.mxo_e8m0.restype = ctypes.c_double
        ci = ctypes.c_int
        lib.mxo_decode.argtypes = [ci, ctypes.c_uint8]
        lib.mxo_decode.restype = ctypes.c_double
        lib.mxo_rows_fmt.argtypes = [i64, i64, i64, u8p, u8p, u8p, u8p, i64, i64p,
                                     f64p, f64p, ci, ci, ci]
        lib.mxo_rows_fmt.restype = ci
        lib.mxo_points_fmt.argtypes = [i64, i64, i64, u8p, u8p, u8p, u8p, i64,
                                       i64p, i64p, f64p, f64p, ci, ci, ci]
        lib.mxo_points_fmt.restype = ci
        lib.mxo_e4m3_rne.argtypes = [ctypes.c_double]
        lib.mxo_e4m3_rne.restype = ctypes.c_uint8
        lib.mxo_quantize_e4m3.argtypes = [i64, i64, f64p, ci, u8p, u8p]
        lib.mxo_quantize_e4m3.restype = ci
        lib.mxo_e4m3_sr.argtypes = [ctypes.c_double, ctypes.c_uint32]
        lib.mxo_e4m3_sr.restype = ctypes.c_uint8
        lib.mxo_quantize_e4m3_sr.argtypes = [i64, i64, f64p, ci, ctypes.c_void_p, u8p, u8p]
        lib.mxo_quantize_e4m3_sr.restype = ci
        lib.mxo_round_f32.argtypes = [ctypes.c_double]
        lib.mxo_round_f32.restype = ctypes.c_float
        lib.mxo_round_bf16.argtypes = [ctypes.c_double]
        lib.mxo_round_bf16.restype = ctypes.c_uint16
        lib.mxo_round_bf16_array.argtypes = [f64p, ctypes.c_void_p, i64]
        lib.mxo_round_bf16_array.restype = None
        _lib = lib
    return _lib


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _u8(x) -> np.ndarray:
    if hasattr(x, "numpy"):  # torch CPU tensor
        x = x.contiguous().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8 codes, got {a.dtype}")
    return a


def e4m3(code: int) -> float:
    """Value of one E4M3 byte (OCP MX v1.0 E4M3)."""
    return _load().mxo_e4m3(int(code) & 0xFF)


# element format ids (OCP MX v1.0 element formats; one code per byte, the
# sub-byte formats in the low bits)
FORMATS = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4}


def decode(fmt: str, code: int) -> float:
    """Value of one element code in format fmt (a key of FORMATS)."""
    return _load().mxo_decode(FORMATS[fmt], int(code) & 0xFF)


def e8m0(code: int) -> float:
    """Value of one E8M0 scale byte: 2**(code-127), NaN for 255."""
    return _load().mxo_e8m0(int(code) & 0xFF)


def _shapes(A, As, B, Bs):
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or K % 32:
        raise ValueError(f"bad shapes A{A.shape} B{B.shape}")
    if As.shape != (M, K // 32) or Bs.shape != (N, K // 32):
        raise ValueError(f"bad scale shapes As{As.shape} Bs{Bs.shape}")
    return M, N, K


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def rows(A, As, B, Bs, rows=None, c_in=None, threads: int | None = None,
         a_fmt: str = "e4m3", b_fmt: str = "e4m3"):
    """Full output rows of the product.  Returns (ref, bound), float64 arrays
    of shape (len(rows), N).  ``rows=None`` means every row.  ``c_in`` (the
    accumulated-into C, any float dtype, shape (len(rows), N)) is added to
    ref and its magnitude to bound when given (use_acc).  ``a_fmt`` and
    ``b_fmt`` name the element formats (keys of FORMATS)."""
    A, As, B, Bs = map(_u8, (A, As, B, Bs))
    M, N, K = _shapes(A, As, B, Bs)
    idx = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    ref = np.empty((idx.size, N), dtype=np.float64)
    bnd = np.empty((idx.size, N), dtype=np.float64)
    rc = _load().mxo_rows_fmt(M, N, K, _ptr(A), _ptr(As), _ptr(B), _ptr(Bs), idx.size,
                              _ptr(idx), _ptr(ref), _ptr(bnd), threads or host_threads(),
                              FORMATS[a_fmt], FORMATS[b_fmt])
    if rc != 0:
        raise ValueError("mxo_rows rejected its arguments")
    if c_in is not None:
        c = np.asarray(c_in, dtype=np.float64).reshape(idx.size, N)
        ref += c
        bnd += np.abs(c)
    return ref, bnd


def points(A, As, B, Bs, I, J, c_in=None, threads: int | None = None,
           a_fmt: str = "e4m3", b_fmt: str = "e4m3"):
    """The product at points (I[p], J[p]).  Returns (ref, bound), float64
    vectors.  ``c_in`` (values of C at those points) is added when given."""
    A, As, B, Bs = map(_u8, (A, As, B, Bs))
    M, N, K = _shapes(A, As, B, Bs)
    I = np.ascontiguousarray(I, dtype=np.int64)
    J = np.ascontiguousarray(J, dtype=np.int64)
    if I.shape != J.shape:
        raise ValueError("I and J differ in shape")
    ref = np.empty(I.size, dtype=np.float64)
    bnd = np.empty(I.size, dtype=np.float64)
    rc = _load().mxo_points_fmt(M, N, K, _ptr(A), _ptr(As), _ptr(B), _ptr(Bs), I.size,
                                _ptr(I), _ptr(J), _ptr(ref), _ptr(bnd), threads or host_threads(),
                                FORMATS[a_fmt], FORMATS[b_fmt])
    if rc != 0:
        raise ValueError("mxo_points rejected its arguments")
    if c_in is not None:
        c = np.asarray(c_in, dtype=np.float64).reshape(I.size)
        ref += c
        bnd += np.abs(c)
    return ref, bnd


def e4m3_rne(y: float) -> int:
    """E4M3 code nearest to y after clamping to +-448, ties to even."""
    return int(_load().mxo_e4m3_rne(float(y)))


def e4m3_sr(y: float, r: int) -> int:
    """E4M3 code of y by stochastic rounding with the random word r: with
    lo <= |y| < lo + q adjacent E4M3 magnitudes (|y| clamped to 448), lo + q
    when r < 2^32 (|y| - lo) / q, else lo; sign kept."""
    return int(_load().mxo_e4m3_sr(float(y), int(r) & 0xFFFFFFFF))


def quantize_e4m3(x, along_cols: bool = False, rand_bits=None):
    """MX quantization of a real R x C matrix (any float dtype, values taken
    exactly) to E4M3 codes with E8M0 scales per 32 values: along each row
    (scales R x C/32) or, with along_cols, down each column (scales
    C x R/32, row j for column j).  The codes round to nearest even, or,
    given rand_bits (R x C uint32, one random word per value), stochastically
    (``e4m3_sr`` of the scaled value as an FP32 number).  Returns (codes
    uint8 R x C, scales)."""
    if hasattr(x, "numpy"):  # torch tensor (bfloat16 and float32 widen exactly)
        x = x.detach().to("cpu").double().numpy()
    xd = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    R, C = xd.shape
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((C, R // 32) if along_cols else (R, C // 32), dtype=np.uint8)
    if rand_bits is None:
        rc = _load().mxo_quantize_e4m3(R, C, _ptr(xd), int(bool(along_cols)), _ptr(codes),
                                       _ptr(scales))
    else:
        if hasattr(rand_bits, "numpy"):
            rand_bits = rand_bits.detach().to("cpu").numpy()
        rb = np.ascontiguousarray(np.asarray(rand_bits).view(np.uint32))
        if rb.shape != (R, C):
            raise ValueError("rand_bits must be R x C")
        rc = _load().mxo_quantize_e4m3_sr(R, C, _ptr(xd), int(bool(along_cols)),
                                          rb.ctypes.data_as(ctypes.c_void_p), _ptr(codes),
                                          _ptr(scales))
    if rc != 0:
        raise ValueError("the oracle's quantizer rejected its arguments")
    return codes, scales


def round_f32(x) -> np.ndarray:
    """Round-to-nearest-even double -> binary32."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even double -> bfloat16, returned as uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().mxo_round_bf16_array(_ptr(x), out.ctypes.data_as(ctypes.c_void_p), x.size)
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (a bfloat16 is the top half of a
    binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def accept(out, ref, bound, out_dtype: str):
    """Per-element acceptance of a computed C against the oracle.

    out_dtype "f32":  |out - ref| <= 1e-5 * bound
    out_dtype "bf16": |out - ref| <= 2^-8 * |ref| + 1e-5 * bound
    with ref the unrounded double result.  Elements whose bound exceeds the
    largest binary32 (the "overflow class": some terms alone exceed the
    output range) are accepted when out is non-finite or within tolerance.
    A non-finite out equal to the rounded reference (same infinity) matches.

    ``out`` is float values (f32) or, for "bf16", either uint16 bit patterns
    or already-decoded values.  Returns a dict of statistics; ``ok`` tells
    whether every element passed.
    """
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    o = np.asarray(out)
    if out_dtype == "bf16" and o.dtype == np.uint16:
        o = bf16_bits_to_f64(o)
    o = o.astype(np.float64).reshape(ref.shape)
    if out_dtype == "f32":
        tol = 1e-5 * bound
    elif out_dtype == "bf16":
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * bound
    else:
        raise ValueError(out_dtype)
    with np.errstate(invalid="ignore", over="ignore"):
        err = np.abs(o - ref)
        within = err <= tol
        ovf = bound > FLT_MAX
        rounded = round_f32(ref).astype(np.float64)
        same_inf = np.isinf(o) & (o == rounded)
        ok_el = within | same_inf | (ovf & ~np.isfinite(o))
        finite_err = np.where(np.isfinite(err) & (bound > 0), err / np.where(bound > 0, bound, 1.0), 0.0)
    bad = ~ok_el
    return {
        "ok": bool(not bad.any()),
        "n": int(ref.size),
        "n_bad": int(bad.sum()),
        "n_overflow_class": int(ovf.sum()),
        "max_err_over_bound": float(finite_err[~ovf].max()) if (~ovf).any() else 0.0,
        "first_bad": (np.argwhere(bad)[0].tolist() if bad.any() else None),
    }
