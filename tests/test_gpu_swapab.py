"""Skinny problems (M <= 128) on the transposed kernel (C^T = B^T x A^T, the
columns of B on the MMA's 128-row side, the rows of A as its N), through the
C interface, against the CPU oracle element by element.

The kernel is chosen automatically for M <= 128 with 8-bit element formats
(MXGEMM_OPT_MODE = 0) and on request (MXGEMM_OPT_MODE = 3).  Cases cover:
the K split inside a cluster (1 to 8 CTAs per 128-column block, chosen by N),
N past a 128-column block, N % 16 != 0 (B re-pitched), K % 128 != 0 and
K % 512 != 0 (scale rows read byte by byte), M not a multiple of 16, use_acc,
BF16 output, packed scales, unaligned scale pointers, mixed E4M3 / E5M2
operands (whose format fields swap in the instruction descriptor), the
timeout path, and the full-size skinny workloads.

Tolerances as in the other parity tests (FP32: 1e-5 * bound; BF16: 2^-8
|ref| + 1e-5 * bound); small integers with unit scales are bit-exact.
"""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")

SWAP = 3


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    handle = mx.mxgemm_create(0)
    mx.mxgemm_set_option(handle, mx.OPT_MODE, SWAP)
    yield handle
    mx.mxgemm_destroy(handle)


@pytest.mark.parametrize("M", [1, 16, 37, 64, 100, 128])
@pytest.mark.parametrize("N", [2304, 8192])
def test_exact_integers_bitwise(h, M, N):
    p = mi.random_problem(M, N, 2048, seed=7 + M + N, kind="int")
    C = gu.run_gpu(h, p)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    got = C.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


def test_row_scales_localised(h):
    # integer data; A's scales depend on the row only (the MMA's B-operand
    # scales): a mis-mapped scale shows up as a wrong power of two in a row
    p = mi.random_problem(100, 512, 512, seed=3, kind="int")
    p.As = (127 + (torch.arange(100) % 7) - 3).to(torch.uint8)[:, None].repeat(1, p.K // 32).contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    bad_rows = np.unique(np.argwhere(C != ref)[:, 0])
    assert bad_rows.size == 0, f"rows with wrong values: {bad_rows[:16].tolist()}"


def test_col_scales_localised(h):
    # B's scales depend on the column only (the MMA's A-operand scales)
    p = mi.random_problem(48, 640, 512, seed=4, kind="int")
    p.Bs = (127 + (torch.arange(640) % 9) - 4).to(torch.uint8)[:, None].repeat(1, p.K // 32).contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    bad_cols = np.unique(np.argwhere(C != ref)[:, 1])
    assert bad_cols.size == 0, f"columns with wrong values: {bad_cols[:16].tolist()}"


def test_kblock_scales_localised(h):
    p = mi.random_problem(64, 256, 1024, seed=5, kind="int")
    kb = torch.arange(p.K // 32)
    p.As = (127 + (kb % 5) - 2).to(torch.uint8)[None, :].repeat(64, 1).contiguous()
    p.Bs = (127 + (kb % 3) - 1).to(torch.uint8)[None, :].repeat(256, 1).contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert np.array_equal(C, ref)


# N picks the K split: 8192 -> 64 blocks x 2, 1024 -> 8 blocks x 8,
# 20096 -> 157 blocks (more than the SMs) x 1; 8240 and 200 end inside a
# block; 1000 and 7000 are not multiples of 16 (B re-pitched)
SHAPES = [(1, 8192, 4096), (16, 8240, 2048), (64, 1024, 4096), (100, 200, 512), (17, 1000, 640),
          (128, 20096, 512), (5, 7000, 480), (33, 4096, 96), (128, 128, 32), (2, 16, 160)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_shapes_against_oracle(h, M, N, K, out_dtype):
    p = mi.random_problem(M, N, K, seed=M * 7 + N + K, kind="normal", out_dtype=out_dtype)
    gu.check_full(h, p)


@pytest.mark.parametrize("M,N,K", [(16, 8192, 2048), (100, 1000, 640), (64, 2304, 4096)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_use_acc(h, M, N, K, out_dtype):
    p = mi.random_problem(M, N, K, seed=11 + M, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, N, 11 + M, out_dtype)
    gu.check_full(h, p, c_init=cin, use_acc=True)


def test_codes_over_all_finite_values(h):
    # every finite E4M3 code (subnormals, zeros, +-448) and scales 120..134
    p = mi.random_problem(64, 4096, 2048, seed=21, kind="codes")
    gu.check_full(h, p)


@pytest.mark.parametrize("fa,fb", [("e5m2", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
def test_mixed_8bit_formats(h, fa, fb):
    # the MMA's A operand is B: the descriptor's two format fields swap
    p = mi.with_formats(mi.random_problem(40, 1536, 1024, seed=31, kind="normal"), fa, fb, seed=31)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, ["e4m3", "e5m2"].index(fa))
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, ["e4m3", "e5m2"].index(fb))
    try:
        C = gu.run_gpu(h, p)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, a_fmt=fa, b_fmt=fb)
    res = oracle.accept(C.cpu().numpy(), ref, bound, "f32")
    assert res["ok"], res


def _shifted(t):
    buf = torch.empty(t.numel() + 16, dtype=torch.uint8, device=gu.DEV)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t.to(gu.DEV))
    assert v.data_ptr() % 16 == 1
    return v


@pytest.mark.parametrize("M,N,K", [(16, 8192, 4096), (100, 1000, 640), (1, 300, 1024)])
def test_scale_sources_bit_identical(h, M, N, K):
    # the scale chunks built from TMA-staged rows (aligned, K % 512 == 0),
    # from byte loads (unaligned pointers) and copied from packed scales give
    # the same C, bit for bit
    p = mi.random_problem(M, N, K, seed=41 + M, kind="normal")
    A, B = p.A.to(gu.DEV), p.B.to(gu.DEV)
    variants = [(p.As.to(gu.DEV), p.Bs.to(gu.DEV), mx.SCALES_ROW_MAJOR),
                (_shifted(p.As), _shifted(p.Bs), mx.SCALES_ROW_MAJOR),
                (mi.pack_scales(p.As).to(gu.DEV), mi.pack_scales(p.Bs, along_cols=True).to(gu.DEV),
                 mx.SCALES_PACKED)]
    outs = []
    try:
        for As, Bs, layout in variants:
            mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, layout)
            C = torch.full((M, N), float("nan"), device=gu.DEV)
            mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, mx.OUT_F32)
            torch.cuda.synchronize()
            assert mx.mxgemm_get_device_status(h)[0] == 0
            outs.append(C.cpu())
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32)), "unaligned scales differ"
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32)), "packed scales differ"
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert oracle.accept(outs[0].numpy(), ref, bound, "f32")["ok"]


def test_auto_mode_and_tiled_path_agree_with_oracle(h):
    # automatic mode takes this kernel for M <= 128; the tiled single-CTA
    # path (mode 1) computes the same product with another summation order:
    # both within tolerance of the oracle
    p = mi.random_problem(48, 2304, 2048, seed=51, kind="normal")
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    try:
        for mode in (0, 1, SWAP):
            mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
            C = gu.run_gpu(h, p)
            res = oracle.accept(C.cpu().numpy(), ref, bound, "f32")
            assert res["ok"], (mode, res)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_MODE, SWAP)


def test_repeat_determinism(h):
    # the K splits are added in a fixed order: identical results run to run
    p = mi.random_problem(16, 8192, 8192, seed=61, kind="codes")
    a = gu.run_gpu(h, p).cpu()
    b = gu.run_gpu(h, p).cpu()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_mode_rejects_what_it_cannot_run(h):
    dev = gu.DEV
    A = torch.zeros((200, 64), dtype=torch.uint8, device=dev)
    S = torch.full((200, 2), 127, dtype=torch.uint8, device=dev)
    B = torch.zeros((64, 16), dtype=torch.uint8, device=dev)
    T = torch.full((16, 2), 127, dtype=torch.uint8, device=dev)
    C = torch.full((200, 16), 5.0, device=dev)
    # more than 128 rows
    assert mx.mxgemm_run(h, 200, 16, 64, A, S, B, T, C, 0, mx.OUT_F32, check=False) == mx.ERR_INVALID_VALUE
    # a 4-bit operand
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 4)
    try:
        st = mx.mxgemm_run(h, 100, 16, 64, A, S, B, T, C, 0, mx.OUT_F32, check=False)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 0)
    assert st == mx.ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)


def test_timeout_reports_and_device_stays_usable():
    # the load-issuing warp issues nothing: the waits run out, the kernel
    # records MXGEMM_ERR_TIMEOUT and returns; the next call is correct again
    from block_scaled_gemm_gb300 import _build
    _build.build()
    g = mx.mxgemm_create(0)
    try:
        mx.mxgemm_set_option(g, mx.OPT_MODE, SWAP)
        p = mi.random_problem(16, 8192, 4096, seed=71, kind="normal")  # two-CTA clusters
        A, As, B, Bs = (t.to(gu.DEV) for t in (p.A, p.As, p.B, p.Bs))
        mx.mxgemm_set_option(g, mx.OPT_WAIT_TIMEOUT_NS, 50_000_000)
        mx.mxgemm_set_option(g, mx.OPT_TEST_STALL_PRODUCER, 1)
        C = torch.zeros((p.M, p.N), device=gu.DEV)
        mx.mxgemm_run(g, p.M, p.N, p.K, A, As, B, Bs, C, 0, mx.OUT_F32)
        st, det = mx.mxgemm_get_device_status(g)
        assert st == mx.ERR_TIMEOUT, (st, det)
        mx.mxgemm_set_option(g, mx.OPT_TEST_STALL_PRODUCER, 0)
        mx.mxgemm_set_option(g, mx.OPT_WAIT_TIMEOUT_NS, 2_000_000_000)
        gu.check_full(g, p)
    finally:
        mx.mxgemm_destroy(g)


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_skinny_workloads_full(h, M):
    # the decode-like workloads at full size, every element
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    try:
        p = mi.skinny(M)
        res, *_ = gu.check_full(h, p)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_MODE, SWAP)
    assert res["max_err_over_bound"] < 1e-5
