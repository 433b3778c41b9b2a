"""The no-allocation entry point, mxgemm_run_noalloc, and its status word.

Some callers cannot allocate device memory at the point where they call the
GEMM: a plug-in whose host framework owns all device memory and hands it only
inputs and outputs, or code that must not allocate once it is running (an
allocation there can fail, stall other streams or fragment the caller's
pool).  This entry point keeps its scratch in a fixed device array instead of
a handle's workspace.  The tests call it through the C interface twice in a
row on each pair of problems, so that the shared scratch is overwritten, and
check every result two ways: against the regular entry point, mxgemm_run, bit
for bit (both run the same single-CTA kernel on whole tiles), and against the
CPU oracle within the parity tolerance of the other GPU tests.

The problems cover B re-pitched into the scratch (N % 16 != 0) and no scratch
at all (N % 16 == 0); scale rows staged by TMA (K a multiple of 512) and read
byte by byte (K = 480); FP32 and BF16 output; and use_acc on a pre-filled C.

The file is named to be collected last, so that a run that stops at the first
failure has already run every other test.
"""
import pytest
import torch

import mx_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")


def _c_start(p, use_acc):
    """C before the call: NaN when use_acc = 0 (ignored), else seeded values."""
    tdt = torch.float32 if p.out_dtype == "f32" else torch.bfloat16
    if use_acc:
        return mi.c_init(p.M, p.N, seed=p.M + p.N, out_dtype=p.out_dtype).to(tdt)
    return torch.full((p.M, p.N), float("nan"), dtype=tdt)


def _noalloc(p, use_acc):
    A, As, B, Bs = (t.to(gu.DEV) for t in (p.A, p.As, p.B, p.Bs))
    C = _c_start(p, use_acc).to(gu.DEV)
    mx.mxgemm_run_noalloc(p.M, p.N, p.K, A, As, B, Bs, C, int(use_acc), gu.out_code(p.out_dtype),
                          torch.cuda.current_stream())
    return C


def _bits(C, out_dtype):
    return C.view(torch.int16) if out_dtype == "bf16" else C.view(torch.int32)


# (problem, use_acc), run back to back in pairs
PROBLEMS = [
    (lambda: mi.random_problem(300, 520, 1024, seed=31, kind="normal", out_dtype="f32"), False),
    (lambda: mi.random_problem(513, 1000, 2048, seed=32, kind="normal", out_dtype="bf16"), False),
    (lambda: mi.random_problem(300, 512, 480, seed=33, kind="normal", out_dtype="f32"), True),
    (lambda: mi.random_problem(257, 1001, 4096, seed=34, kind="normal", out_dtype="bf16"), False),
]


@pytest.mark.parametrize("pair", [(0, 1), (2, 3)])
def test_noalloc_matches_regular_entry_point_and_oracle_twice(pair):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    cases = [(PROBLEMS[i][0](), PROBLEMS[i][1]) for i in pair]
    # two no-allocation calls in a row, back to back on the stream
    outs = [_noalloc(p, ua) for p, ua in cases]
    st, det = mx.mxgemm_noalloc_get_status(torch.cuda.current_stream())
    assert st == 0, (st, det)
    h = mx.mxgemm_create(0)
    # whole single-CTA tiles, as the no-allocation path computes them
    mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 0)
    mx.mxgemm_set_option(h, mx.OPT_MODE, 1)
    try:
        for (p, ua), c_na in zip(cases, outs):
            c0 = _c_start(p, ua)
            c_reg = gu.run_gpu(h, p, c_init=c0, use_acc=ua)
            cin = c0.to(torch.float64).numpy() if ua else None
            ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, c_in=cin)
            res = oracle.accept(gu.to_numpy_out(c_na, p.out_dtype), ref, bound, p.out_dtype)
            assert res["ok"], f"{p.name} (use_acc={ua}) against the oracle: {res}"
            assert torch.equal(_bits(c_na, p.out_dtype), _bits(c_reg, p.out_dtype)), \
                f"{p.name} (use_acc={ua}): not bit-identical to mxgemm_run"
    finally:
        mx.mxgemm_destroy(h)


def test_noalloc_timeout_is_reported_then_clean():
    # The load-issuing warp is told to issue nothing, so the kernel's bounded
    # waits run out (50 ms) and it records MXGEMM_ERR_TIMEOUT in the
    # no-allocation status word, drains and returns; nothing traps.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = mi.random_problem(256, 256, 256, seed=35, kind="normal")
    stream = torch.cuda.current_stream()
    assert mx.mxgemm_noalloc_get_status(stream)[0] == 0
    try:
        mx.mxgemm_noalloc_set_option(mx.OPT_WAIT_TIMEOUT_NS, 50_000_000)
        mx.mxgemm_noalloc_set_option(mx.OPT_TEST_STALL_PRODUCER, 1)
        _noalloc(p, False)
        st, det = mx.mxgemm_noalloc_get_status(stream)
        assert st == mx.ERR_TIMEOUT, (st, det)
        assert det != 0
        # the read cleared the word
        assert mx.mxgemm_noalloc_get_status(stream) == (0, 0)
    finally:
        mx.mxgemm_noalloc_set_option(mx.OPT_TEST_STALL_PRODUCER, 0)
        mx.mxgemm_noalloc_set_option(mx.OPT_WAIT_TIMEOUT_NS, 2_000_000_000)
    # hook off: a correct result and a clean status again
    C = _noalloc(p, False)
    assert mx.mxgemm_noalloc_get_status(stream)[0] == 0
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    res = oracle.accept(C.cpu().numpy(), ref, bound, "f32")
    assert res["ok"], res


def test_noalloc_options_validated():
    assert mx.library().mxgemm_noalloc_set_option(mx.OPT_MODE, 1) == mx.ERR_INVALID_VALUE
    assert mx.library().mxgemm_noalloc_set_option(mx.OPT_WAIT_TIMEOUT_NS, 0) == mx.ERR_INVALID_VALUE
    assert mx.library().mxgemm_noalloc_set_option(mx.OPT_TEST_STALL_PRODUCER, 2) == mx.ERR_INVALID_VALUE


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
