"""GPU parity: the CUDA path (through the C interface) against the CPU oracle,
element by element, on seeded inputs.

Tolerances (per element, ref = unrounded double oracle value, bound =
sum_k |a_k b_k| with scales):
    FP32 out: |C - ref| <= 1e-5 * bound
    BF16 out: |C - ref| <= 2^-8 |ref| + 1e-5 * bound
Small integers with unit scales must be bit-exact (FP32 partial sums of
integers below 2^24 are exact in any order).
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
    yield handle
    mx.mxgemm_destroy(handle)


def _mode(h, m):
    mx.mxgemm_set_option(h, mx.OPT_MODE, m)


# ---------------------------------------------------------------- exactness

@pytest.mark.parametrize("mode", [1, 2])
def test_exact_integers_bitwise(h, mode):
    _mode(h, mode)
    p = mi.random_problem(384, 512, 1024, seed=2, kind="int")
    C = gu.run_gpu(h, p)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    got = C.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("mode", [1, 2])
def test_row_scales_localised(h, mode):
    # integer data, A scale depends on the row only: a mis-mapped scale lane
    # shows up as a wrong power of two in that row
    _mode(h, mode)
    p = mi.random_problem(256, 256, 256, seed=3, kind="int")
    As = (127 + (torch.arange(256) % 7) - 3).to(torch.uint8)[:, None].repeat(1, p.K // 32)
    p.As = As.contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    bad_rows = np.unique(np.argwhere(C != ref)[:, 0])
    assert bad_rows.size == 0, f"rows with wrong values: {bad_rows[:16].tolist()}"


@pytest.mark.parametrize("mode", [1, 2])
def test_col_scales_localised(h, mode):
    _mode(h, mode)
    p = mi.random_problem(256, 512, 256, seed=4, kind="int")
    p.Bs = (127 + (torch.arange(512) % 9) - 4).to(torch.uint8)[:, None].repeat(1, p.K // 32).contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    bad_cols = np.unique(np.argwhere(C != ref)[:, 1])
    assert bad_cols.size == 0, f"columns with wrong values: {bad_cols[:16].tolist()}"


@pytest.mark.parametrize("mode", [1, 2])
def test_kblock_scales_localised(h, mode):
    _mode(h, mode)
    p = mi.random_problem(256, 256, 512, seed=5, kind="int")
    kb = torch.arange(p.K // 32)
    p.As = (127 + (kb % 5) - 2).to(torch.uint8)[None, :].repeat(256, 1).contiguous()
    p.Bs = (127 + (kb % 3) - 1).to(torch.uint8)[None, :].repeat(256, 1).contiguous()
    C = gu.run_gpu(h, p).cpu().numpy().astype(np.float64)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert np.array_equal(C, ref)


# ---------------------------------------------------------------- tolerance parity

@pytest.mark.parametrize("mode", [1, 2])
def test_square_256(h, mode):
    _mode(h, mode)
    p = mi.square_256()
    res, *_ = gu.check_full(h, p)
    assert res["max_err_over_bound"] < 1e-5


SIZES = [1, 31, 127, 128, 129, 255, 257]
KS = [32, 96, 128, 160, 4096]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("K", KS)
def test_small_sweep_f32(h, mode, K):
    _mode(h, mode)
    for i, M in enumerate(SIZES):
        N = SIZES[(i * 3 + 2) % len(SIZES)]
        p = mi.random_problem(M, N, K, seed=100 + i + K, kind="normal")
        gu.check_full(h, p)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_use_acc(h, mode, out_dtype):
    _mode(h, mode)
    p = mi.random_problem(300, 520, 384, seed=7, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(p.M, p.N, 7, out_dtype)
    gu.check_full(h, p, c_init=cin, use_acc=True)
    # use_acc = 0 ignores C (NaN-filled by run_gpu)
    gu.check_full(h, p, c_init=None, use_acc=False)


@pytest.mark.parametrize("mode", [1, 2])
def test_bf16_out_and_ragged_n(h, mode):
    _mode(h, mode)
    # N not a multiple of 16: the B rows are re-pitched internally; N not a
    # multiple of 8: the BF16 epilogue takes its scalar path
    for (M, N, K) in [(200, 1000, 256), (129, 77, 160), (64, 4100, 128)]:
        for od in ("f32", "bf16"):
            p = mi.random_problem(M, N, K, seed=M + N, kind="normal", out_dtype=od)
            gu.check_full(h, p)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_one_vs_two_cta_identical(h, out_dtype):
    # Whole tiles in both modes (no tail splitting): every output element is
    # the same sequence of K = 32 block-scaled MMAs, accumulated in FP32 in
    # the same order, whether its 128 rows belong to a single-CTA MMA
    # (M = 128) or to one half of a pair's MMA (M = 256).  The two results
    # must agree bit for bit, and each with the oracle.
    p = mi.random_problem(512, 768, 1024, seed=11, kind="normal", out_dtype=out_dtype)
    mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 0)
    try:
        _mode(h, 1)
        c1 = gu.run_gpu(h, p).cpu()
        _mode(h, 2)
        c2 = gu.run_gpu(h, p).cpu()
    finally:
        mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 1)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert oracle.accept(gu.to_numpy_out(c1, out_dtype), ref, bound, out_dtype)["ok"]
    assert oracle.accept(gu.to_numpy_out(c2, out_dtype), ref, bound, out_dtype)["ok"]
    bits = (lambda c: c.view(torch.int16)) if out_dtype == "bf16" else (lambda c: c.view(torch.int32))
    assert torch.equal(bits(c1), bits(c2))


def test_repeat_determinism(h):
    _mode(h, 0)
    p = mi.random_problem(640, 512, 2048, seed=12, kind="codes")
    a = gu.run_gpu(h, p).cpu()
    b = gu.run_gpu(h, p).cpu()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_degenerate_sizes(h):
    _mode(h, 0)
    dev = gu.DEV
    A = torch.zeros((4, 64), dtype=torch.uint8, device=dev)
    S = torch.full((4, 2), 127, dtype=torch.uint8, device=dev)
    B = torch.zeros((64, 8), dtype=torch.uint8, device=dev)
    T = torch.full((8, 2), 127, dtype=torch.uint8, device=dev)
    C = torch.full((4, 8), 5.0, device=dev)
    # M == 0 / N == 0: no-op
    mx.mxgemm_run(h, 0, 8, 64, A, S, B, T, C, 0, mx.OUT_F32)
    mx.mxgemm_run(h, 4, 0, 64, A, S, B, T, C, 0, mx.OUT_F32)
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)
    # K == 0: use_acc keeps C, otherwise C = 0
    mx.mxgemm_run(h, 4, 8, 0, A, S, B, T, C, 1, mx.OUT_F32)
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)
    mx.mxgemm_run(h, 4, 8, 0, A, S, B, T, C, 0, mx.OUT_F32)
    torch.cuda.synchronize()
    assert torch.all(C == 0.0)


def test_invalid_arguments_rejected_before_launch(h):
    dev = gu.DEV
    A = torch.zeros((4, 64), dtype=torch.uint8, device=dev)
    S = torch.full((4, 2), 127, dtype=torch.uint8, device=dev)
    B = torch.zeros((64, 16), dtype=torch.uint8, device=dev)
    T = torch.full((16, 2), 127, dtype=torch.uint8, device=dev)
    C = torch.full((4, 16), 5.0, device=dev)
    st = mx.mxgemm_run(h, 4, 16, 48, A, S, B, T, C, 0, mx.OUT_F32, check=False)
    assert st == mx.ERR_INVALID_VALUE  # K % 32 != 0
    st = mx.mxgemm_run(h, 4, 16, 64, A, S, B, T, C, 0, 7, check=False)
    assert st == mx.ERR_INVALID_VALUE  # bad dtype
    st = mx.mxgemm_run(h, 4, 16, 64, A.data_ptr() + 1, S, B, T, C, 0, mx.OUT_F32, check=False)
    assert st == mx.ERR_MISALIGNED
    st = mx.mxgemm_run(h, 4, 16, 64, None, S, B, T, C, 0, mx.OUT_F32, check=False)
    assert st == mx.ERR_INVALID_VALUE
    host = torch.zeros((4, 64), dtype=torch.uint8)
    st = mx.mxgemm_run(h, 4, 16, 64, host, S, B, T, C, 0, mx.OUT_F32, check=False)
    assert st == mx.ERR_INVALID_VALUE  # not device memory
    st = mx.mxgemm_run(h, -1, 16, 64, A, S, B, T, C, 0, mx.OUT_F32, check=False)
    assert st == mx.ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)


def test_timeout_reports_and_device_stays_usable():
    # the load-issuing warp is told to issue nothing: the consumers' waits run
    # out, the kernel records MXGEMM_ERR_TIMEOUT, drains and returns
    from block_scaled_gemm_gb300 import _build
    _build.build()
    g = mx.mxgemm_create(0)
    try:
        for mode in (1, 2):
            mx.mxgemm_set_option(g, mx.OPT_MODE, mode)
            mx.mxgemm_set_option(g, mx.OPT_WAIT_TIMEOUT_NS, 50_000_000)
            mx.mxgemm_set_option(g, mx.OPT_TEST_STALL_PRODUCER, 1)
            p = mi.random_problem(256, 256, 256, seed=21, kind="normal")
            A, As, B, Bs = (t.to(gu.DEV) for t in (p.A, p.As, p.B, p.Bs))
            C = torch.zeros((256, 256), device=gu.DEV)
            mx.mxgemm_run(g, 256, 256, 256, A, As, B, Bs, C, 0, mx.OUT_F32)
            st, det = mx.mxgemm_get_device_status(g)
            assert st == mx.ERR_TIMEOUT, (st, det)
            # the same handle, hook off: correct results again
            mx.mxgemm_set_option(g, mx.OPT_TEST_STALL_PRODUCER, 0)
            mx.mxgemm_set_option(g, mx.OPT_WAIT_TIMEOUT_NS, 2_000_000_000)
            gu.check_full(g, p)
    finally:
        mx.mxgemm_destroy(g)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("out_dtype,use_acc", [("f32", False), ("bf16", False), ("f32", True), ("bf16", True)])
def test_stream_k_tail_matches_whole_tiles(h, mode, out_dtype, use_acc):
    # 256 x 22016 x 8192: 172 tiles of 128x256 (86 of 256x256) with 64 K
    # steps, one full wave on 152 CTAs (76 pairs), then a tail of 20 (10)
    # tiles -- the last 10 tile columns -- whose K ranges are split over all
    # CTAs and finished by the CTA holding each tile's last K steps.  Checked
    # on 16 whole rows against the oracle, with the tail on and off.
    _mode(h, mode)
    p = mi.random_problem(256, 256 * 86, 8192, seed=41 + mode, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(p.M, p.N, 41, out_dtype) if use_acc else None
    rows = np.array([0, 1, 31, 64, 127, 128, 129, 160, 191, 200, 223, 250, 253, 254, 255, 100])
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows,
                             c_in=None if cin is None else cin.to(torch.float64).numpy()[rows])
    outs = {}
    try:
        for sk in (1, 0):
            mx.mxgemm_set_option(h, mx.OPT_STREAM_K, sk)
            C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
            outs[sk] = gu.to_numpy_out(C, out_dtype)
            res = oracle.accept(outs[sk][rows], ref, bound, out_dtype)
            assert res["ok"], f"stream_k={sk}: {res}"
    finally:
        mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 1)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("out_dtype,use_acc", [("f32", False), ("bf16", False), ("f32", True), ("bf16", True)])
def test_half_width_tail(h, mode, out_dtype, use_acc):
    # 2560 x 3976 x 512: 160 tiles of 256x256 (320 of 128x256), two full
    # waves on 76 pairs (152 CTAs), then 8 (16) leftover tiles -- rows
    # 2048..2559, tile columns 12..15 -- each computed as two 128-column
    # halves, the last half holding only 8 columns.  Whole rows in and
    # outside that region are checked against the oracle.
    _mode(h, mode)
    p = mi.random_problem(2560, 3976, 512, seed=51 + mode, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(p.M, p.N, 51, out_dtype) if use_acc else None
    rows = np.array([0, 5, 2047, 2048, 2100, 2175, 2176, 2300, 2303, 2304, 2431, 2432, 2559])
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows,
                             c_in=None if cin is None else cin.to(torch.float64).numpy()[rows])
    C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
    res = oracle.accept(gu.to_numpy_out(C, out_dtype)[rows], ref, bound, out_dtype)
    assert res["ok"], res


@pytest.mark.parametrize("mode", [1, 2])
def test_half_width_only(h, mode):
    # 2000 x 1000 x 256: fewer tiles than half the CTAs (pairs), so every
    # tile is computed as two 128-column halves; full check.
    _mode(h, mode)
    p = mi.random_problem(2000, 1000, 256, seed=61 + mode, kind="normal", out_dtype="f32")
    gu.check_full(h, p)


CLC_CASES = [
    # (M, N, K, out_dtype, use_acc): fewer clusters than fit (no cancel succeeds),
    # many more (most items taken by cancelling), a half-width tail, ragged edges
    (256, 256, 4096, "f32", False),
    (4096, 4096, 1024, "f32", False),
    (2560, 3976, 512, "bf16", False),
    (1000, 1000, 1024, "f32", True),
]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", CLC_CASES, ids=lambda c: "x".join(map(str, c[:3])) + f"-{c[3]}-acc{int(c[4])}")
def test_clc_scheduler(h, mode, case):
    # Cluster launch control: one cluster per work item, the running ones
    # cancel launches and take their items.  Checked against the oracle on
    # whole rows spread over the tiles, and bit for bit against the static
    # schedule (each tile is computed by one CTA or pair either way).
    M, N, K, out_dtype, use_acc = case
    _mode(h, mode)
    p = mi.random_problem(M, N, K, seed=71 + mode + M, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, N, 71, out_dtype) if use_acc else None
    rows = np.unique(np.linspace(0, M - 1, 24).astype(int))
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, rows=rows,
                             c_in=None if cin is None else cin.to(torch.float64).numpy()[rows])
    outs = {}
    try:
        for sched in (1, 0):
            mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, sched)
            C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
            outs[sched] = gu.to_numpy_out(C, out_dtype)
            res = oracle.accept(outs[sched][rows], ref, bound, out_dtype)
            assert res["ok"], f"scheduler={sched}: {res}"
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, 0)
    assert np.array_equal(outs[0].view(np.uint32) if out_dtype == "f32" else outs[0],
                          outs[1].view(np.uint32) if out_dtype == "f32" else outs[1])


@pytest.mark.parametrize("mode", [1, 2])
def test_clc_scheduler_full_check(h, mode):
    # every element of a problem whose items are mostly taken by cancelling
    _mode(h, mode)
    p = mi.random_problem(1536, 2304, 256, seed=81 + mode, kind="normal", out_dtype="f32")
    try:
        mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, 1)
        gu.check_full(h, p)
    finally:
        mx.mxgemm_set_option(h, mx.OPT_SCHEDULER, 0)


@pytest.mark.parametrize("M", [1, 16, 100, 128])
@pytest.mark.parametrize("out_dtype,use_acc", [("f32", False), ("bf16", True)])
def test_skinny_split_k(h, M, out_dtype, use_acc):
    # The tiled single-CTA path (mode 1; automatic mode takes the transposed
    # kernel for these shapes) with at most 128 rows and fewer tiles than
    # CTAs: every tile's K steps are split over all CTAs, with partial sums
    # of the valid rows only.  Full check against the oracle, and against
    # whole tiles (tail balancing off).
    _mode(h, 1)
    p = mi.random_problem(M, 2304, 2048, seed=101 + M, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, p.N, 101, out_dtype) if use_acc else None
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs,
                             c_in=None if cin is None else cin.to(torch.float64).numpy())
    try:
        for sk in (1, 0):
            mx.mxgemm_set_option(h, mx.OPT_STREAM_K, sk)
            C = gu.run_gpu(h, p, c_init=cin, use_acc=use_acc)
            res = oracle.accept(gu.to_numpy_out(C, out_dtype), ref, bound, out_dtype)
            assert res["ok"], f"stream_k={sk}: {res}"
    finally:
        mx.mxgemm_set_option(h, mx.OPT_STREAM_K, 1)


def test_plan_cache_churn_and_workspace_growth(h):
    # more distinct problems than the handle caches plans for, cycled twice
    # without synchronizing between calls, growing and reusing the workspace
    # (stream-ordered); every result checked against the oracle
    _mode(h, 0)
    shapes = [(64, 96, 64), (300, 520, 256), (1000, 200, 512), (129, 1000, 1024), (520, 520, 2048),
              (2048, 64, 320), (17, 4000, 128), (700, 700, 640), (256, 4096, 512), (1500, 300, 96),
              (33, 65, 8192), (900, 1300, 160)]
    probs = [mi.random_problem(M, N, K, seed=300 + i, kind="normal", out_dtype="f32" if i % 3 else "bf16")
             for i, (M, N, K) in enumerate(shapes)]
    dev = [tuple(t.to(gu.DEV) for t in (p.A, p.As, p.B, p.Bs)) for p in probs]
    outs = []
    stream = torch.cuda.current_stream()
    for rnd in range(2):
        for p, (A, As, B, Bs) in zip(probs, dev):
            tdt = torch.float32 if p.out_dtype == "f32" else torch.bfloat16
            C = torch.full((p.M, p.N), float("nan"), dtype=tdt, device=gu.DEV)
            mx.mxgemm_run(h, p.M, p.N, p.K, A, As, B, Bs, C, 0, gu.out_code(p.out_dtype), stream)
            outs.append((p, C))
    torch.cuda.synchronize()
    st, det = mx.mxgemm_get_device_status(h)
    assert st == 0, (st, det)
    for p, C in outs:
        ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
        res = oracle.accept(gu.to_numpy_out(C, p.out_dtype), ref, bound, p.out_dtype)
        assert res["ok"], f"{p.name}: {res}"


@pytest.mark.parametrize("mode,M", [(1, 300), (2, 300), (1, 100), (0, 100)])
@pytest.mark.parametrize("K", [1024, 384, 160])
def test_scales_at_unaligned_addresses(h, mode, M, K):
    # A_scale and B_scale one byte past a 16-byte boundary: the scale chunks
    # are built from byte loads instead of 16-byte ones (M = 300: the repack,
    # for single CTAs and pairs; M = 100, mode 1: the tiled kernel's scale
    # loader, mode 0: the transposed kernel's scale builder, both reading
    # rows byte by byte also when K % 512 != 0); the result is the same, bit
    # for bit
    _mode(h, mode)
    p = mi.random_problem(M, 520, K, seed=K + mode + M, kind="normal")
    ref_c = gu.run_gpu(h, p).cpu()
    dev = gu.DEV

    def unaligned(t):
        buf = torch.empty(t.numel() + 16, dtype=torch.uint8, device=dev)
        v = buf[1:1 + t.numel()].view(t.shape)
        v.copy_(t.to(dev))
        assert v.data_ptr() % 16 == 1
        return v

    A, B = p.A.to(dev), p.B.to(dev)
    As, Bs = unaligned(p.As), unaligned(p.Bs)
    C = torch.full((p.M, p.N), float("nan"), dtype=torch.float32, device=dev)
    mx.mxgemm_run(h, p.M, p.N, K, A, As, B, Bs, C, 0, mx.OUT_F32)
    torch.cuda.synchronize()
    assert mx.mxgemm_get_device_status(h)[0] == 0
    assert torch.equal(C.cpu().view(torch.int32), ref_c.view(torch.int32))
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert oracle.accept(C.cpu().numpy(), ref, bound, "f32")["ok"]
