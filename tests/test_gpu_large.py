"""Problems past 2^31 elements: C of the GEMM, or the quantizer's input,
holds more than 2^31 elements, so every linear index past that mark must be
formed in 64 bits.  Checked against the oracle at sampled points, most of
them past the mark (the sizes are far beyond what the oracle computes
whole).  About 20 GB of device memory at most.

- tiled kernel, pairs and single CTAs: 65664 x 32784 x 64 (2.15e9 elements
  of C, ragged against the 256-wide tiles), FP32 and BF16 output;
- transposed skinny kernel: 128 x (2^24 + 32) x 32;
- quantizer, FP32 and BF16 input, blocks along rows and down columns:
  65536 x 32800 (mx_inputs.pattern_matrix, exact in both input types).
"""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")

MARK = 2 ** 31


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    handle = mx.mxgemm_create(0)
    yield handle
    mx.mxgemm_destroy(handle)


def _sample(M, N, n=512, seed=0):
    """Linear indices: most past 2^31, some anywhere, the mark and the last."""
    g = np.random.default_rng(seed)
    lin = np.concatenate([g.integers(MARK, M * N, 3 * n // 4), g.integers(0, M * N, n // 4),
                          [MARK, MARK - 1, M * N - 1]])
    return lin // N, lin % N


@pytest.mark.parametrize("mode,M,N,K", [(2, 65664, 32784, 64), (1, 65664, 32784, 64),
                                        (0, 128, 2 ** 24 + 32, 32)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_c_past_2g_elements(h, mode, M, N, K, out_dtype):
    assert M * N > MARK
    p = mi.random_problem(M, N, K, seed=M % 97 + N % 89, kind="int", out_dtype=out_dtype)
    mx.mxgemm_set_option(h, mx.OPT_MODE, mode)
    try:
        C = gu.run_gpu(h, p)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_MODE, 0)
    I, J = _sample(M, N)
    got = C[torch.as_tensor(I, device=C.device), torch.as_tensor(J, device=C.device)]
    got = got.float().cpu().numpy().astype(np.float64)
    del C
    torch.cuda.empty_cache()
    ref, bound = oracle.points(p.A, p.As, p.B, p.Bs, I, J)
    if out_dtype == "f32":
        # small integers with unit scales: exact in any summation order
        assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} of {got.size} points differ"
    else:
        res = oracle.accept(got, ref, bound, "bf16")
        assert res["ok"], res


@pytest.fixture(scope="module")
def big_x():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    R, C = 65536, 32800
    assert R * C > MARK
    x = mi.pattern_matrix(R, C, device="cuda")
    yield x
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("along_cols", [False, True])
def test_quantizer_past_2g_elements(big_x, x_dtype, along_cols):
    R, C = big_x.shape
    X = big_x if x_dtype == "f32" else big_x.to(torch.bfloat16)
    codes = torch.empty((R, C), dtype=torch.uint8, device=X.device)
    scales = torch.empty((C, R // 32) if along_cols else (R, C // 32), dtype=torch.uint8, device=X.device)
    mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=along_cols)
    torch.cuda.synchronize()
    # the last 32-row block lies wholly past 2^31 elements (row 65474 starts
    # past it); and the first block for comparison
    for r0 in (R - 32, 0):
        rows = list(range(r0, r0 + 32))
        xr = mi.pattern_matrix(R, C, rows=rows)  # the same values, on the CPU
        if x_dtype == "bf16":
            xr = xr.to(torch.bfloat16)
        rc, rs = oracle.quantize_e4m3(xr, along_cols=along_cols)
        got_c = codes[r0:r0 + 32].cpu().numpy()
        got_s = (scales[:, r0 // 32:r0 // 32 + 1] if along_cols else scales[r0:r0 + 32]).cpu().numpy()
        assert np.array_equal(got_c, rc), f"rows {r0}..: {np.count_nonzero(got_c != rc)} codes differ"
        assert np.array_equal(got_s, rs), f"rows {r0}..: {np.count_nonzero(got_s != rs)} scales differ"
    del X, codes, scales
    torch.cuda.empty_cache()
