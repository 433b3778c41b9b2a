"""Randomized parity sweep: seeded random shapes, tile modes, output types, scale
layouts (row-major, row-major at unaligned addresses, packed),
use_acc, element formats and schedulers, each checked against the oracle on
whole rows (including the first and last row and a row from every 256-row
band touched), so that interior tiles, ragged edges and the tail-balancing
paths (half-width tiles, stream-K, skinny split) are all exercised."""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")

FORMATS = ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"]


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    handle = mx.mxgemm_create(0)
    yield handle
    mx.mxgemm_destroy(handle)


def _case(i):
    rng = np.random.default_rng(1000 + i)
    kind = rng.integers(0, 4)
    if kind == 0:      # small and ragged
        M, N = int(rng.integers(1, 700)), int(rng.integers(1, 900))
        K = 32 * int(rng.integers(1, 40))
    elif kind == 1:    # skinny
        M, N = int(rng.integers(1, 129)), int(rng.integers(256, 3000))
        K = 128 * int(rng.integers(8, 40))
    elif kind == 2:    # a few waves with a tail
        M, N = int(rng.integers(1500, 3100)), int(rng.integers(1500, 3100))
        K = 128 * int(rng.integers(2, 12))
    else:              # long K after a full wave (stream-K territory)
        M, N = 2560, 2048 + 256 * int(rng.integers(0, 3))
        K = 128 * int(rng.integers(64, 72))
    mode = int(rng.integers(0, 3))
    out_dtype = "f32" if rng.random() < 0.6 else "bf16"
    use_acc = bool(rng.random() < 0.3)
    fa = FORMATS[0] if rng.random() < 0.6 else FORMATS[int(rng.integers(0, 5))]
    fb = FORMATS[0] if rng.random() < 0.6 else FORMATS[int(rng.integers(0, 5))]
    sched = int(rng.random() < 0.2)
    return M, N, K, mode, out_dtype, use_acc, fa, fb, sched


@pytest.mark.parametrize("i", range(40))
def test_random_configuration(h, i):
    M, N, K, mode, out_dtype, use_acc, fa, fb, sched = _case(i)
    g = torch.Generator().manual_seed(2000 + i)
    p = mi.random_problem(M, N, K, seed=3000 + i, kind="normal", out_dtype=out_dtype)
    if (fa, fb) != ("e4m3", "e4m3"):
        p = mi.with_formats(p, fa, fb, seed=4000 + i)
    cin = mi.c_init(M, N, 5000 + i, out_dtype) if use_acc else None
    rows = sorted(set([0, M - 1] + list(range(min(M - 1, 137), M, 256)) +
                      torch.randint(0, M, (6,), generator=g).tolist()))
    rows = np.array(rows[:24], dtype=np.int64)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows, a_fmt=fa, b_fmt=fb,
                             c_in=None if cin is None else cin.to(torch.float64).numpy()[rows])
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, FORMATS.index(fa))
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FORMATS.index(fb))
    mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, sched)
    try:
        C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
        mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, 0)
        mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, 0)
    res = oracle.accept(gu.to_numpy_out(C, out_dtype)[rows], ref, bound, out_dtype)
    assert res["ok"], f"case {i} {(M, N, K, mode, out_dtype, use_acc, fa, fb, sched)}: {res}"


def _shifted(t):
    # the same bytes one past a 16-byte boundary
    buf = torch.empty(t.numel() + 16, dtype=torch.uint8, device="cuda")
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("i", range(24))
def test_random_scale_layouts(h, i):
    # the same random problem with aligned row-major scales, row-major scales
    # at unaligned addresses and packed scales: identical C, bit for bit, and
    # the oracle on sampled rows
    M, N, K, mode, out_dtype, use_acc, _, _, _ = _case(100 + i)
    p = mi.random_problem(M, N, K, seed=6000 + i, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, N, 7000 + i, out_dtype) if use_acc else None
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    A, B = p.A.cuda(), p.B.cuda()
    variants = [(p.As.cuda(), p.Bs.cuda(), mx.SCALES_ROW_MAJOR),
                (_shifted(p.As.cuda()), _shifted(p.Bs.cuda()), mx.SCALES_ROW_MAJOR),
                (mi.pack_scales(p.As).cuda(), mi.pack_scales(p.Bs, along_cols=True).cuda(), mx.SCALES_PACKED)]
    outs = []
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    try:
        for As, Bs, layout in variants:
            mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, layout)
            C = (cin.to(tdt).cuda().clone() if cin is not None
                 else torch.full((M, N), float("nan"), dtype=tdt, device="cuda"))
            mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, int(use_acc), gu.out_code(out_dtype))
            torch.cuda.synchronize()
            st, det = mx.mxgemm_get_device_status(h)
            assert st == 0, (st, det)
            outs.append(C.cpu())
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_ROW_MAJOR)
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    iv = torch.int16 if out_dtype == "bf16" else torch.int32
    assert torch.equal(outs[0].view(iv), outs[1].view(iv)), "unaligned scales differ"
    assert torch.equal(outs[0].view(iv), outs[2].view(iv)), "packed scales differ"
    rows = np.unique(np.array([0, M - 1, M // 2, min(M - 1, 129)], dtype=np.int64))
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows,
                             c_in=None if cin is None else cin.to(torch.float64).numpy()[rows])
    res = oracle.accept(gu.to_numpy_out(outs[0], out_dtype)[rows], ref, bound, out_dtype)
    assert res["ok"], (M, N, K, mode, res)
