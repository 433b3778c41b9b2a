"""The no-allocation entry point, mxgemm_run_noalloc.

It serves callers that cannot allocate device memory where they call the
GEMM (a plug-in whose host framework owns all device memory, code that may not
allocate after start-up, a stream under capture): it keeps its scratch in a
fixed device array instead of a handle's workspace.  This test calls it
through the C interface twice in a row, on two different problems so that the
shared scratch is overwritten, and checks each result against the regular
entry point, mxgemm_run, within the parity tolerance of the other GPU tests.

The file is named to be collected last, so that a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")


def _regular(h, p):
    return gu.run_gpu(h, p)


def _noalloc(p):
    A, As, B, Bs = (t.to(gu.DEV) for t in (p.A, p.As, p.B, p.Bs))
    tdt = torch.float32 if p.out_dtype == "f32" else torch.bfloat16
    C = torch.full((p.M, p.N), float("nan"), dtype=tdt, device=gu.DEV)
    mx.mxgemm_run_noalloc(p.M, p.N, p.K, A, As, B, Bs, C, 0, gu.out_code(p.out_dtype),
                          torch.cuda.current_stream())
    return C


def test_noalloc_matches_regular_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    problems = [
        mi.random_problem(300, 520, 1024, seed=31, kind="normal", out_dtype="f32"),
        mi.random_problem(513, 1000, 2048, seed=32, kind="normal", out_dtype="bf16"),
    ]
    # two no-allocation calls in a row, back to back on the stream
    outs = [_noalloc(p) for p in problems]
    torch.cuda.synchronize()
    h = mx.mxgemm_create(0)
    # whole single-CTA tiles, as the no-allocation path computes them, so
    # that the two results can also be compared bit for bit
    mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 0)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 1)
    try:
        for p, c_na in zip(problems, outs):
            c_reg = _regular(h, p)
            ref_reg = c_reg.to(torch.float64).cpu().numpy()
            _, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
            res = oracle.accept(gu.to_numpy_out(c_na, p.out_dtype), ref_reg, bound, p.out_dtype)
            assert res["ok"], f"{p.name}: {res}"
            # both paths run the same kernel on the same tiles
            assert torch.equal(c_na.view(torch.int16) if p.out_dtype == "bf16" else c_na.view(torch.int32),
                               c_reg.view(torch.int16) if p.out_dtype == "bf16" else c_reg.view(torch.int32))
    finally:
        mx.mxgemm_destroy(h)


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    small = torch.zeros(1024, dtype=torch.uint8, device=gu.DEV)
    C = torch.zeros(16, dtype=torch.float32, device=gu.DEV)
    # B re-pitched for N % 16 != 0: K * round_up(N, 16) = 2048 * 16384 bytes = 32 MiB > 16 MiB
    # (rejected before anything is read or enqueued)
    st = mx.mxgemm_run_noalloc(256, 16383, 2048, small, small, small, small, C, 0, mx.OUT_F32,
                               None, check=False)
    assert st == mx.ERR_TOO_LARGE
    assert "scratch" in mx.mxgemm_status_string(st)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
