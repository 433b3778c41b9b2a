"""GPU parity at the full sizes of the five standard workloads, in the launch
configuration the benchmark uses.  The square, long-K and ragged workloads
are checked on every element; for the MLP shape (1.9e12 multiply-adds) whole
rows and columns (first, last, tile edges, random) plus random points are
checked, each against the oracle computed one output at a time."""
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
    yield handle
    mx.mxgemm_destroy(handle)


def _sampled_check(p, C, out_dtype, n_rows=24, n_cols=24, n_rand=20000, seed=0, c_in=None):
    got = gu.to_numpy_out(C, out_dtype)
    rows, cols, ri, rj = gu.sample_points(p.M, p.N, n_rows, n_cols, n_rand, seed)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows,
                             c_in=None if c_in is None else c_in[rows])
    r1 = oracle.accept(got[rows], ref, bound, out_dtype)
    assert r1["ok"], f"{p.name} rows: {r1}"
    I = np.repeat(np.arange(p.M), cols.size)
    J = np.tile(cols, p.M)
    ref, bound = oracle.points(p.A, p.As, p.B, p.Bs, I, J,
                               c_in=None if c_in is None else c_in[I, J])
    r2 = oracle.accept(got[I, J], ref, bound, out_dtype)
    assert r2["ok"], f"{p.name} cols: {r2}"
    ref, bound = oracle.points(p.A, p.As, p.B, p.Bs, ri, rj,
                               c_in=None if c_in is None else c_in[ri, rj])
    r3 = oracle.accept(got[ri, rj], ref, bound, out_dtype)
    assert r3["ok"], f"{p.name} points: {r3}"
    return r1, r2, r3


def test_square_4096_full(h):
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    p = mi.square_4096()
    res, *_ = gu.check_full(h, p)
    assert res["max_err_over_bound"] < 1e-5


@pytest.mark.parametrize("mode", [1, 2])
def test_square_4096_tile_modes_sampled(h, mode):
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    p = mi.square_4096()
    C = gu.run_gpu(h, p)
    _sampled_check(p, C, "f32", n_rows=8, n_cols=8, n_rand=5000)


def test_mlp_up_pair_mode_bf16(h):
    # LLM MLP up-projection, BF16 out, CTA-pair mode
    mx.mxgemm_set_option(h, mx.OPT_MODE, 2)
    p = mi.mlp_up()
    C = gu.run_gpu(h, p)
    _sampled_check(p, C, "bf16")


def test_longk_chained_use_acc_full(h):
    # K = 65536 as 4 calls of 16384 accumulated into one FP32 C (zero-filled),
    # compared element by element with the single K = 65536 sum (the whole
    # 2048 x 2048 matrix; about 20 s of oracle on 16 host cores)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    p = mi.longk()
    gu.check_full(h, p, c_init=torch.zeros((p.M, p.N)), use_acc=True)


def test_longk_first_call_ignores_nan_c(h):
    # variant: C starts NaN, the first call has use_acc = 0
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    p = mi.longk()
    C = gu.run_gpu(h, p, c_init=None, use_acc=False)
    _sampled_check(p, C, "f32", n_rows=8, n_cols=8, n_rand=2000, seed=3)


def test_ragged_edges_extreme_scales_full(h):
    # the whole 5000 x 7000 matrix (about 25 s of oracle on 16 host cores)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    p = mi.ragged()
    gu.check_full(h, p)


@pytest.mark.parametrize("mode", [1, 2])
def test_ragged_tile_modes(h, mode):
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    p = mi.ragged()
    C = gu.run_gpu(h, p)
    _sampled_check(p, C, "f32", n_rows=8, n_cols=8, n_rand=5000, seed=mode)
