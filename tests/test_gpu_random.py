"""Randomized parity sweep: seeded random shapes, tile modes, output types,
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
