"""B given transposed, N x K with K contiguous (MXGEMM_OPT_B_MAJOR =
MXGEMM_B_N_BY_K: the layout of a linear layer's weight), through the C
interface, against the CPU oracle on the same product: the oracle takes B
as K x N, the GPU its transpose.

Covers every tile mode (single CTAs, CTA pairs, the transposed skinny
kernel), the tails (half-width tiles, stream-K), N that is not a multiple of
16 (no re-pitch pass is needed in this layout), use_acc and BF16 output,
6- and 4-bit B in both element layouts, packed scales and the host-buffer
entry point.  Small integers with unit scales must be bit-exact.
"""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    handle = mx.mxgemm_create(0)
    mx.mxgemm_set_option(handle, mx.OPT_B_MAJOR, mx.B_N_BY_K)
    yield handle
    mx.mxgemm_destroy(handle)


def _run(h, p, mode, c_init=None, use_acc=False, out_dtype=None):
    """Run problem p with B passed as its N x K transpose; returns C (GPU)."""
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    q = mi.Problem(p.name, p.M, p.N, p.K, p.A, p.As, p.B.t().contiguous(), p.Bs, p.out_dtype, p.use_acc)
    return gu.run_gpu(h, q, c_init=c_init, use_acc=use_acc, out_dtype=out_dtype)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_exact_integers_bitwise(h, mode):
    M = 100 if mode == 3 else 384
    p = mi.random_problem(M, 520, 1024, seed=2, kind="int")
    C = _run(h, p, mode)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    got = C.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} mismatches"


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_col_scales_localised(h, mode):
    # B's scales depend on the column (row of the transposed B) only
    M = 64 if mode == 3 else 256
    p = mi.random_problem(M, 640, 512, seed=4, kind="int")
    p.Bs = (127 + (torch.arange(640) % 9) - 4).to(torch.uint8)[:, None].repeat(1, p.K // 32).contiguous()
    C = _run(h, p, mode).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    bad_cols = np.unique(np.argwhere(C != ref)[:, 1])
    assert bad_cols.size == 0, f"columns with wrong values: {bad_cols[:16].tolist()}"


SHAPES = [(300, 1000, 512), (257, 7000, 1024), (1024, 1024, 2048), (513, 4096, 8192),
          (640, 768, 4096), (16, 8192, 4096), (100, 1000, 640), (1, 777, 96)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shapes_against_oracle(h, mode, M, N, K):
    # mode 0 picks pairs for M > 128 and the transposed kernel for M <= 128;
    # the shapes include half-width tails (few tiles), stream-K tails
    # (K = 8192 after full waves) and N % 16 != 0
    if mode in (1, 2) and M <= 128:
        pytest.skip("the transposed kernel's shapes run under mode 0")
    p = mi.random_problem(M, N, K, seed=M + N + K + mode, kind="normal")
    C = _run(h, p, mode)
    rows = np.unique(np.array([0, M - 1, M // 2, min(M - 1, 129)], dtype=np.int64))
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows)
    res = oracle.accept(C.cpu().numpy()[rows], ref, bound, "f32")
    assert res["ok"], res


@pytest.mark.parametrize("mode,M", [(1, 300), (2, 300), (3, 64)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_use_acc_full(h, mode, M, out_dtype):
    p = mi.random_problem(M, 520, 768, seed=9 + M, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, 520, 9, out_dtype)
    C = _run(h, p, mode, c_init=cin, use_acc=True)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, c_in=cin.to(torch.float64).numpy())
    res = oracle.accept(gu.to_numpy_out(C, out_dtype), ref, bound, out_dtype)
    assert res["ok"], res


@pytest.mark.parametrize("mode", [1, 2])
def test_same_result_as_k_by_n(h, mode):
    # the two layouts of B feed the same products to the tensor cores
    p = mi.random_problem(512, 768, 2048, seed=31, kind="normal")
    c_nk = _run(h, p, mode).cpu()
    mx.mxgemm_set_option(h, mx.OPT_B_MAJOR, mx.B_K_BY_N)
    try:
        c_kn = gu.run_gpu(h, p).cpu()
    finally:
        mx.mxgemm_set_option(h, mx.OPT_B_MAJOR, mx.B_N_BY_K)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    for c in (c_nk, c_kn):
        assert oracle.accept(c.numpy(), ref, bound, "f32")["ok"]


BITS = {"e2m3": 6, "e3m2": 6, "e2m1": 4}
FMT = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4}


@pytest.mark.parametrize("fb", ["e2m1", "e3m2", "e5m2"])
@pytest.mark.parametrize("packed", [False, True])
def test_formats_of_b(h, fb, packed):
    # sub-byte B in this layout: groups of 16 along K (packed by the library
    # per call, or already packed); E5M2 as an 8-bit check
    M, N, K = 300, 1000, 1024
    p = mi.with_formats(mi.random_problem(M, N, K, seed=FMT[fb], kind="normal"), "e4m3", fb, seed=FMT[fb])
    bt = p.B.t().contiguous()
    if packed and fb in BITS:
        bt = mi.pack_elements(bt, BITS[fb])
    q = mi.Problem(p.name, M, N, K, p.A, p.As, bt, p.Bs, "f32", False)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 2)
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FMT[fb])
    mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_PACKED if packed else mx.ELEMS_BYTE)
    try:
        C = gu.run_gpu(h, q)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_BYTE)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, b_fmt=fb)
    res = oracle.accept(C.cpu().numpy(), ref, bound, "f32")
    assert res["ok"], res


def test_packed_scales(h):
    p = mi.random_problem(700, 1300, 1024, seed=41, kind="normal")
    A, B = p.A.to(gu.DEV), p.B.t().contiguous().to(gu.DEV)
    As, Bs = mi.pack_scales(p.As).to(gu.DEV), mi.pack_scales(p.Bs, along_cols=True).to(gu.DEV)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_PACKED)
    try:
        C = torch.full((p.M, p.N), float("nan"), device=gu.DEV)
        mx.mxgemm_run(h, p.M, p.N, p.K, A, As, B, Bs, C, 0, mx.OUT_F32)
        torch.cuda.synchronize()
        assert mx.mxgemm_get_device_status(h)[0] == 0
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert oracle.accept(C.cpu().numpy(), ref, bound, "f32")["ok"]


def test_host_entry_point(h):
    # the host-buffer entry point copies B as it is given (N x K)
    p = mi.random_problem(700, 520, 1024, seed=51, kind="normal")
    hA, hAs, hBs = (t.contiguous().pin_memory() for t in (p.A, p.As, p.Bs))
    hB = p.B.t().contiguous().pin_memory()
    C = torch.full((p.M, p.N), float("nan"), dtype=torch.float32).pin_memory()
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    stream = torch.cuda.current_stream()
    mx.mxgemm_run_host(h, p.M, p.N, p.K, hA, hAs, hB, hBs, C, 0, mx.OUT_F32, stream)
    torch.cuda.synchronize()
    assert mx.mxgemm_get_device_status(h)[0] == 0
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert oracle.accept(C.numpy(), ref, bound, "f32")["ok"]


def test_option_rejects_unknown_values(h):
    with pytest.raises(mx.MxgemmError):
        mx.mxgemm_set_option(h, mx.OPT_B_MAJOR, 2)
