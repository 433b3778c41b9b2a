"""NaN inputs through the C interface: E4M3 codes 0x7F / 0xFF and the E8M0
scale byte 255 are NaN (OCP MX v1.0; the readings of the pages take the
same).  A NaN element or scale of A must make its row of C NaN, one of B its
column, and every other element must be what it is without them (small
integers with unit scales: exact).  C starts zeroed, so a NaN can only come
from the kernel.  Single CTAs, CTA pairs and the transposed skinny kernel,
FP32 and BF16 output."""
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


@pytest.mark.parametrize("mode,M", [(1, 300), (2, 300), (3, 100)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_nan_inputs_poison_exactly_their_rows_and_columns(h, mode, M, out_dtype):
    N, K = 520, 256
    p = mi.random_problem(M, N, K, seed=13 + mode, kind="int", out_dtype=out_dtype)
    ref0, bound0 = oracle.rows(p.A, p.As, p.B, p.Bs)
    nan_rows = [5, 77, M // 2]
    nan_cols = [100, 400]
    p.A = p.A.clone()
    p.As = p.As.clone()
    p.B = p.B.clone()
    p.Bs = p.Bs.clone()
    p.A[5, 17] = 0x7F
    p.A[77, 200] = 0xFF
    p.As[M // 2, 3] = 255
    p.B[33, 100] = 0x7F
    p.Bs[400, 6] = 255
    mask = np.zeros((M, N), dtype=bool)
    mask[nan_rows, :] = True
    mask[:, nan_cols] = True
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert np.array_equal(np.isnan(ref), mask)  # the oracle's own reading
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    try:
        C = gu.run_gpu(h, p, c_init=torch.zeros((M, N)), use_acc=False)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    got = C.float().cpu().numpy().astype(np.float64)
    bad_nan = np.argwhere(np.isnan(got) != mask)
    assert bad_nan.size == 0, f"NaN pattern differs at {bad_nan[:8].tolist()}"
    res = oracle.accept(got[~mask], ref0[~mask], bound0[~mask], out_dtype)
    assert res["ok"], res
    if out_dtype == "f32":
        assert np.array_equal(got[~mask], ref0[~mask])
