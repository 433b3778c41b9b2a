"""Scales in the packed layout (the order the tensor cores read them):
mxgemm_quantize_ex writes them and a run with OPT_SCALE_LAYOUT =
SCALES_PACKED reads them without a repack prepass.  The packed scales must
hold exactly the row-major scales (checked by unpacking them here, with the
layout of mxgemm.h written out independently), and a run on packed scales
must give the same C, bit for bit, as the same run on row-major scales, in
every tile mode and through the host-buffer entry point."""
import numpy as np
import pytest
import torch

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
    yield handle
    mx.mxgemm_destroy(handle)


def _unpack(P, n, kbn, cols):
    """Row-major n x kbn scales from packed bytes (A rows, or B columns)."""
    S = -(-kbn // 4)
    r = np.arange(n)[:, None]
    kb = np.arange(kbn)[None, :]
    inner = (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    if cols:
        at = (((r // 256) * S + kb // 4) * 2 + (r // 128) % 2) * 512 + inner
    else:
        at = ((r // 128) * S + kb // 4) * 512 + inner
    return P[at]


def _quantize(x, along_cols, layout):
    R, C = x.shape
    X = x.cuda()
    codes = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    nbytes = mx.mxgemm_scale_bytes(R, C, along_cols, layout)
    scales = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN until written
    mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=along_cols, scale_layout=layout)
    torch.cuda.synchronize()
    return codes, scales


@pytest.mark.parametrize("along_cols,R,C", [(False, 300, 416), (False, 128, 1024), (False, 1, 32),
                                            (True, 416, 300), (True, 1024, 520), (True, 32, 1)])
def test_packed_quantizer_holds_the_row_major_scales(along_cols, R, C):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = torch.Generator().manual_seed(R + C)
    x = torch.randn((R, C), generator=g) * torch.exp(torch.randn((R, 1), generator=g) * 4)
    c_rm, s_rm = _quantize(x, along_cols, mx.SCALES_ROW_MAJOR)
    c_pk, s_pk = _quantize(x, along_cols, mx.SCALES_PACKED)
    assert torch.equal(c_rm, c_pk)
    n, kbn = (C, R // 32) if along_cols else (R, C // 32)
    rm = s_rm.cpu().numpy().reshape(n, kbn)
    pk = s_pk.cpu().numpy()
    assert np.array_equal(_unpack(pk, n, kbn, along_cols), rm)
    # every other byte of the packed area is padding, 127
    used = np.zeros(pk.size, dtype=bool)
    r = np.arange(n)[:, None]
    kb = np.arange(kbn)[None, :]
    S = -(-kbn // 4)
    inner = (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    at = ((((r // 256) * S + kb // 4) * 2 + (r // 128) % 2) * 512 + inner) if along_cols else \
        (((r // 128) * S + kb // 4) * 512 + inner)
    used[at.ravel()] = True
    assert np.all(pk[~used] == 127)
    # and the row-major scales are the oracle's
    rc, rs = oracle.quantize_e4m3(x, along_cols=along_cols)
    assert np.array_equal(rm, rs) and np.array_equal(c_rm.cpu().numpy(), rc)


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((M, K), generator=g)
    b = torch.randn((K, N), generator=g) * 0.05
    A, As = _quantize(a, False, mx.SCALES_ROW_MAJOR)
    _, Asp = _quantize(a, False, mx.SCALES_PACKED)
    B, Bs = _quantize(b, True, mx.SCALES_ROW_MAJOR)
    _, Bsp = _quantize(b, True, mx.SCALES_PACKED)
    return A, As.view(M, K // 32), Asp, B, Bs.view(N, K // 32), Bsp


def _run(h, M, N, K, A, As, B, Bs, layout, mode):
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, layout)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    try:
        mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, mx.OUT_F32)
        torch.cuda.synchronize()
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    assert mx.mxgemm_get_device_status(h)[0] == 0
    return C.cpu()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 520, 1024), (700, 1000, 416), (64, 1536, 2048), (1, 264, 4096),
                                   (512, 768, 8192)])
def test_run_on_packed_scales_matches_row_major(h, mode, M, N, K):
    A, As, Asp, B, Bs, Bsp = _operands(M, N, K, seed=M * 3 + N + K)
    c_rm = _run(h, M, N, K, A, As, B, Bs, mx.SCALES_ROW_MAJOR, mode)
    c_pk = _run(h, M, N, K, A, Asp, B, Bsp, mx.SCALES_PACKED, mode)
    assert torch.equal(c_rm.view(torch.int32), c_pk.view(torch.int32))
    ref, bound = oracle.rows(A.cpu().numpy(), As.cpu().numpy(), B.cpu().numpy(), Bs.cpu().numpy())
    assert oracle.accept(c_pk.numpy(), ref, bound, "f32")["ok"]


def test_host_entry_on_packed_scales(h):
    M, N, K = 1000, 520, 1024
    A, As, Asp, B, Bs, Bsp = _operands(M, N, K, seed=77)
    c_dev = _run(h, M, N, K, A, Asp, B, Bsp, mx.SCALES_PACKED, 0)
    hA, hAsp, hB, hBsp = (t.cpu().pin_memory() for t in (A, Asp, B, Bsp))
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_PACKED)
    try:
        mx.mxgemm_run_host(h, M, N, K, hA, hAsp, hB, hBsp, hC, 0, mx.OUT_F32)
        torch.cuda.synchronize()
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
    assert mx.mxgemm_get_device_status(h)[0] == 0
    assert torch.equal(hC.view(torch.int32), c_dev.view(torch.int32))


def test_packed_scales_need_alignment(h):
    M, N, K = 128, 256, 256
    A, As, Asp, B, Bs, Bsp = _operands(M, N, K, seed=5)
    buf = torch.empty(Asp.numel() + 16, dtype=torch.uint8, device="cuda")
    mis = buf[1:1 + Asp.numel()]
    mis.copy_(Asp)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_PACKED)
    try:
        st = mx.mxgemm_run(h, M, N, K, A, mis, B, Bsp, C, 0, mx.OUT_F32, check=False)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
    assert st == mx.ERR_MISALIGNED
    assert mx.library().mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, 2) == mx.ERR_INVALID_VALUE
