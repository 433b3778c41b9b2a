"""Helpers shared by the GPU tests: move a Problem to the GPU, run it through
the C interface, and check the result against the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_gemm_gb300 as mx
import oracle

DEV = torch.device("cuda:0")


def out_code(out_dtype: str) -> int:
    return mx.OUT_F32 if out_dtype == "f32" else mx.OUT_BF16


def to_numpy_out(C: torch.Tensor, out_dtype: str) -> np.ndarray:
    if out_dtype == "f32":
        return C.cpu().numpy()
    return C.cpu().view(torch.int16).numpy().view(np.uint16)


def run_gpu(h, p, c_init: torch.Tensor | None = None, use_acc: bool | None = None,
            out_dtype: str | None = None, stream=None) -> torch.Tensor:
    """Run problem p (all k_chunks calls) and return C on the GPU."""
    use_acc = p.use_acc if use_acc is None else use_acc
    out_dtype = p.out_dtype if out_dtype is None else out_dtype
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    if c_init is None:
        C = torch.full((p.M, p.N), float("nan"), dtype=tdt, device=DEV)
    else:
        C = c_init.to(device=DEV, dtype=tdt).contiguous().clone()
    for c in range(p.k_chunks):
        if p.k_chunks == 1:
            A, As, B, Bs, K = p.A, p.As, p.B, p.Bs, p.K
        else:
            A, As, B, Bs, K = p.chunk(c)
        A, As, B, Bs = (t.to(DEV) for t in (A, As, B, Bs))
        ua = use_acc if c == 0 else True
        mx.mxgemm_run(h, p.M, p.N, K, A, As, B, Bs, C, ua, out_code(out_dtype), stream)
    torch.cuda.synchronize()
    st, det = mx.mxgemm_get_device_status(h)
    assert st == 0, f"device status {st} ({mx.mxgemm_status_string(st)}), detail {det:#x}"
    return C


def check_full(h, p, c_init=None, use_acc=None, out_dtype=None):
    use_acc = p.use_acc if use_acc is None else use_acc
    out_dtype = p.out_dtype if out_dtype is None else out_dtype
    C = run_gpu(h, p, c_init, use_acc, out_dtype)
    cin = None
    if use_acc and c_init is not None:
        cin = c_init.to(torch.float64).numpy()
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs, c_in=cin)
    res = oracle.accept(to_numpy_out(C, out_dtype), ref, bound, out_dtype)
    assert res["ok"], f"{p.name}: {res}"
    return res, C, ref, bound


def sample_points(M: int, N: int, n_rows: int, n_cols: int, n_rand: int, seed: int = 0):
    """Indices for a sampled check: a few full rows and columns (first, last,
    tile edges and random ones) plus random points."""
    g = np.random.default_rng(seed)
    rows = sorted(set([0, M - 1, min(127, M - 1), min(128, M - 1), min(255, M - 1), min(256, M - 1)]
                      + g.integers(0, M, n_rows).tolist()))
    cols = sorted(set([0, N - 1, min(127, N - 1), min(128, N - 1), min(255, N - 1), min(256, N - 1)]
                      + g.integers(0, N, n_cols).tolist()))
    ri = g.integers(0, M, n_rand)
    rj = g.integers(0, N, n_rand)
    return np.array(rows), np.array(cols), ri, rj
