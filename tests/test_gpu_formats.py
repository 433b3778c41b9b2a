"""The other element formats of the scaled MMA (E5M2, E2M3, E3M2, E2M1, and
mixed A/B formats) through the C interface, element by element against the
oracle.  6- and 4-bit operands are given one element per byte (code in the
low bits) and packed on the GPU into the MMA's 16-elements-per-16-bytes form
before the GEMM; ragged N exercises that packing together with the row
re-pitch."""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")

FMT = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4}
BITS = {"e2m3": 6, "e3m2": 6, "e2m1": 4}


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    handle = mx.mxgemm_create(0)
    yield handle
    mx.mxgemm_destroy(handle)


def _codes(fmt, shape, g, junk_high_bits=False):
    if fmt in BITS:
        c = torch.randint(0, 1 << BITS[fmt], shape, generator=g, dtype=torch.int32)
        if junk_high_bits:   # the bits above the code are ignored
            c |= torch.randint(0, 256 >> BITS[fmt], shape, generator=g, dtype=torch.int32) << BITS[fmt]
        return c.to(torch.uint8)
    c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8)
    if fmt == "e4m3":
        c[(c & 0x7F) == 0x7F] = 0x3F
    else:
        c[(c & 0x7C) == 0x7C] = 0x3C
    return c


def _run(h, mode, fa, fb, M, N, K, out_dtype="f32", use_acc=False, seed=0, junk=False):
    g = torch.Generator().manual_seed(seed)
    A = _codes(fa, (M, K), g, junk)
    B = _codes(fb, (K, N), g, junk)
    As = torch.randint(118, 137, (M, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    Bs = torch.randint(118, 137, (N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    p = mi.Problem(f"{fa}x{fb}", M, N, K, A, As, B, Bs, out_dtype, use_acc)
    cin = mi.c_init(M, N, seed, out_dtype) if use_acc else None
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, FMT[fa])
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FMT[fb])
    try:
        C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
    ref, bound = oracle.rows(A, As, B, Bs, a_fmt=fa, b_fmt=fb,
                             c_in=None if cin is None else cin.to(torch.float64).numpy())
    res = oracle.accept(gu.to_numpy_out(C, out_dtype), ref, bound, out_dtype)
    assert res["ok"], f"{fa} x {fb} mode {mode}: {res}"


PAIRS = [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e2m3", "e2m3"), ("e3m2", "e3m2"),
         ("e2m1", "e2m1"), ("e2m1", "e4m3"), ("e4m3", "e2m1"), ("e2m3", "e2m1"), ("e3m2", "e5m2")]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("fa,fb", PAIRS)
def test_formats_full_check(h, mode, fa, fb):
    _run(h, mode, fa, fb, 300, 520, 512, seed=FMT[fa] * 7 + FMT[fb])


@pytest.mark.parametrize("fa,fb", [("e2m1", "e2m1"), ("e3m2", "e2m3"), ("e5m2", "e4m3")])
def test_formats_bf16_use_acc_and_high_bits(h, fa, fb):
    _run(h, 0, fa, fb, 513, 777, 1024, out_dtype="bf16", use_acc=True, seed=3, junk=True)


def test_format_option_rejects_unknown_values(h):
    for opt in (mx.OPT_A_FORMAT, mx.OPT_B_FORMAT):
        with pytest.raises(mx.MxgemmError):
            mx.mxgemm_set_option(h, opt, 5)
        with pytest.raises(mx.MxgemmError):
            mx.mxgemm_set_option(h, opt, -1)


SUB_PAIRS = [("e2m1", "e2m1"), ("e2m3", "e3m2"), ("e3m2", "e4m3"), ("e4m3", "e2m1"), ("e2m1", "e5m2")]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("fa,fb", SUB_PAIRS)
def test_packed_elements_match_byte_elements(h, mode, fa, fb):
    # 6- and 4-bit operands given already in the tensor cores' packed form
    # (MXGEMM_ELEMS_PACKED, read as they are) and one code per byte (packed
    # by the library first): the same C bit for bit, and the oracle on every
    # element
    M, N, K = 300, 528, 1024
    g = torch.Generator().manual_seed(FMT[fa] * 11 + FMT[fb] + mode)
    A = _codes(fa, (M, K), g, junk_high_bits=True)
    B = _codes(fb, (K, N), g, junk_high_bits=True)
    As = torch.randint(118, 137, (M, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    Bs = torch.randint(118, 137, (N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    Ap = mi.pack_elements(A, BITS[fa]) if fa in BITS else A
    Bp = mi.pack_elements(B, BITS[fb]) if fb in BITS else B
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, FMT[fa])
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FMT[fb])
    outs = []
    try:
        for layout, a, b in ((mx.ELEMS_BYTE, A, B), (mx.ELEMS_PACKED, Ap, Bp)):
            mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, layout)
            n0 = mx.mxgemm_get_launch_count(h)
            p = mi.Problem(f"{fa}x{fb}", M, N, K, a, As, b, Bs, "f32", False)
            outs.append((gu.run_gpu(h, p).cpu(), mx.mxgemm_get_launch_count(h) - n0))
    finally:
        mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_BYTE)
        mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    (c_byte, n_byte), (c_packed, n_packed) = outs
    assert torch.equal(c_byte.view(torch.int32), c_packed.view(torch.int32))
    # no packing pass over A or B for packed elements
    assert n_packed == n_byte - (fa in BITS) - (fb in BITS), (n_byte, n_packed)
    ref, bound = oracle.rows(A, As, B, Bs, a_fmt=fa, b_fmt=fb)
    res = oracle.accept(c_packed.numpy(), ref, bound, "f32")
    assert res["ok"], res


def test_packed_elements_need_whole_groups_of_b(h):
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FMT["e2m1"])
    mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_PACKED)
    try:
        dev = gu.DEV
        A = torch.zeros((256, 64), dtype=torch.uint8, device=dev)
        S = torch.full((256, 2), 127, dtype=torch.uint8, device=dev)
        B = torch.zeros((64, 40), dtype=torch.uint8, device=dev)
        T = torch.full((40, 2), 127, dtype=torch.uint8, device=dev)
        C = torch.full((256, 40), 5.0, device=dev)
        st = mx.mxgemm_run(h, 256, 40, 64, A, S, B, T, C, 0, mx.OUT_F32, check=False)
        assert st == mx.ERR_INVALID_VALUE
        with pytest.raises(mx.MxgemmError):
            mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, 2)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_BYTE)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
