"""mxgemm_run_host: operands and result in host memory, through the C
interface.  B and its scales are copied once; the rows of A and C move in
slabs through two device slots while the slabs' GEMMs run.  Results are
checked element by element against the oracle, with pinned and pageable host
buffers, FP32 and BF16 output, use_acc, one slab and many slabs, and two
calls in a row on one handle (the slots and the staging area are reused)."""
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


def _host_run(h, p, pinned, use_acc=False, c_init=None):
    def host(t):
        t = t.contiguous()
        return t.pin_memory() if pinned else t.clone()
    A, As, B, Bs = (host(t) for t in (p.A, p.As, p.B, p.Bs))
    tdt = torch.float32 if p.out_dtype == "f32" else torch.bfloat16
    if c_init is not None:
        C = host(c_init.to(tdt))
    else:
        C = host(torch.full((p.M, p.N), float("nan"), dtype=tdt))
    stream = torch.cuda.current_stream()
    mx.mxgemm_run_host(h, p.M, p.N, p.K, A, As, B, Bs, C, use_acc, gu.out_code(p.out_dtype), stream)
    stream.synchronize()
    st, det = mx.mxgemm_get_device_status(h)
    assert st == 0, (st, det)
    return C


def _check(p, C, cin=None):
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, c_in=None if cin is None else cin.to(torch.float64).numpy())
    res = oracle.accept(gu.to_numpy_out(C, p.out_dtype), ref, bound, p.out_dtype)
    assert res["ok"], res


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("shape,out_dtype,use_acc", [
    ((1000, 600, 512), "f32", False),    # 4 slabs of 256 rows, the last one 232
    ((700, 520, 256), "bf16", True),     # 3 slabs, C read back in
    ((100, 300, 128), "f32", False),     # one slab
    ((2100, 264, 1024), "f32", True),    # 5 slabs of 512 rows
])
def test_run_host_matches_oracle(h, pinned, shape, out_dtype, use_acc):
    M, N, K = shape
    p = mi.random_problem(M, N, K, seed=91 + M, kind="normal", out_dtype=out_dtype)
    cin = mi.c_init(M, N, 91, out_dtype) if use_acc else None
    C = _host_run(h, p, pinned, use_acc, cin)
    _check(p, C, cin)


def test_run_host_twice_and_matches_device_entry(h):
    # two different problems back to back on one handle, then the first
    # again against the device-pointer entry point
    p1 = mi.random_problem(1300, 700, 640, seed=95, kind="normal", out_dtype="f32")
    p2 = mi.random_problem(600, 1100, 384, seed=96, kind="normal", out_dtype="bf16")
    C1 = _host_run(h, p1, True)
    C2 = _host_run(h, p2, True)
    _check(p1, C1)
    _check(p2, C2)
    Cd = gu.run_gpu(h, p1).cpu()
    ref, bound = oracle.rows(p1.A, p1.As, p1.B, p1.Bs)
    assert oracle.accept(Cd.numpy(), ref, bound, "f32")["ok"]


def test_run_host_rejects_bad_arguments(h):
    z = torch.zeros(64, dtype=torch.uint8)
    C = torch.zeros(16, dtype=torch.float32)
    assert mx.mxgemm_run_host(h, 4, 4, 40, z, z, z, z, C, 0, mx.OUT_F32, None, check=False) == mx.ERR_INVALID_VALUE
    assert mx.mxgemm_run_host(h, 4, 4, 32, None, z, z, z, C, 0, mx.OUT_F32, None, check=False) == mx.ERR_INVALID_VALUE
    assert mx.mxgemm_run_host(h, 4, 4, 32, z, z, z, z, C, 0, 7, None, check=False) == mx.ERR_INVALID_VALUE
    # K == 0 zeroes C without use_acc
    C.fill_(3.0)
    assert mx.mxgemm_run_host(h, 4, 4, 0, z, z, z, z, C, 0, mx.OUT_F32, None, check=False) == mx.OK
    assert torch.all(C == 0)


def test_run_host_back_to_back_calls_overlap_correctly(h):
    # consecutive calls overlap on the copy streams (one call's B copy runs
    # while the previous call's last slabs come back); four different
    # problems, each with its own host C, enqueued without synchronizing
    probs = [mi.random_problem(1100, 640, 384, seed=200 + i, kind="normal", out_dtype="f32")
             for i in range(4)]
    outs = []
    stream = torch.cuda.current_stream()
    for p in probs:
        A, As, B, Bs = (t.contiguous().pin_memory() for t in (p.A, p.As, p.B, p.Bs))
        C = torch.full((p.M, p.N), float("nan"), dtype=torch.float32).pin_memory()
        mx.mxgemm_run_host(h, p.M, p.N, p.K, A, As, B, Bs, C, 0, mx.OUT_F32, stream)
        outs.append((A, As, B, Bs, C))
    stream.synchronize()
    for p, (_, _, _, _, C) in zip(probs, outs):
        _check(p, C)


def test_run_host_use_acc_chain_on_one_host_c(h):
    # C accumulated over two K halves by two calls on the same host C, with
    # no synchronization between them: the second call must read the first
    # call's result
    M, N, K = 700, 520, 1024
    p = mi.random_problem(M, N, K, seed=210, kind="normal", out_dtype="f32")
    C = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    halves = []
    for c in range(2):
        k0, k1 = c * K // 2, (c + 1) * K // 2
        A = p.A[:, k0:k1].contiguous().pin_memory()
        As = p.As[:, k0 // 32:k1 // 32].contiguous().pin_memory()
        B = p.B[k0:k1].contiguous().pin_memory()
        Bs = p.Bs[:, k0 // 32:k1 // 32].contiguous().pin_memory()
        halves.append((A, As, B, Bs))
        mx.mxgemm_run_host(h, M, N, K // 2, A, As, B, Bs, C, c, mx.OUT_F32, stream)
    stream.synchronize()
    _check(p, C)
