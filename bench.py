#!/usr/bin/env python3
"""Benchmark of the GB300 MX block-scaled FP8 GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mx|reference]

One step = one C = A.B call through the C interface (scale repack prepass +
the tcgen05 GEMM kernel) on the LLM MLP up-projection workload: M = 8192
tokens, N = 28672, K = 8192, A from N(0,1) activations with 0.1 % outliers
x50, B from N(0, 0.02) weights, both quantized per 32-element K block to E4M3
with E8M0 scales, BF16 output, CTA-pair (cta_group::2) tiles; inputs resident
in HBM.  The operands (311 MB) exceed the 126 MB L2; a buffer of twice the
L2 size is written between timed steps all the same, outside the CUDA events
that time each step on the launching stream.

Prints one JSON line: metric TFLOP/s = 2MNK / t (whole job; t the sum of the
per-step event times), per-step medians (flushed and hot L2), the roofline
of the GEMM kernel (timed alone by events the library records around its
launch) against the MXFP8 tensor peak, a sustained rate (the same step back
to back for a few seconds), the other workloads of the suite in a
"workloads" object (square 4096, long K, ragged, square 256, the skinny
decode shapes with their HBM GB/s), each with its own spot parity,
end-to-end TFLOP/s through the host-buffer entry point with pinned host
buffers (H2D of A, B and scales + D2H of C inside the timed region), SM
clocks sampled during the timed region, and the CPU oracle timed on a bounded
sample of the same workload.

``--impl reference`` times the CPU oracle (the plain FP64 definition) on the
same workload, a bounded sample of rows per step, on the host cores.

Under torchrun (N > 1) every rank runs its own independent GEMM (replicas,
no data exchange); value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "MXFP8 GEMM TFLOP/s (2MNK/t) and % of GB300 dense MXFP8 peak, 1 GPU"
UNIT = "TFLOP/s"
WORKLOAD = "mlp_up_8192x28672x8192"
# the other workloads measured in the same run (the "workloads" object)
WORKLOAD_TABLE = ["square_4096", "longk_2048_65536", "ragged_5000x7000x8192", "square_256",
                  "skinny_1x8192x8192", "skinny_16x8192x8192", "skinny_64x8192x8192",
                  "skinny_128x8192x8192"]
FP8_OVER_BF16 = 2.0  # nominal dense MXFP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
FALLBACK_BF16_BURST = 1900.0  # TFLOP/s, used only when MEASURED_PEAKS.json is absent
FORMATS = ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"]  # C interface order (mxgemm_format_t)
FALLBACK_HBM_GBS = 6800.0     # GB/s, used only when MEASURED_PEAKS.json is absent
KERNEL_SOURCES = ["block_scaled_gemm_gb300/csrc/mxgemm_kernel.cuh",
                  "block_scaled_gemm_gb300/csrc/ptx.cuh"]
PROFILES = ROOT / "profiles"


# ----------------------------------------------------------------------------- ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, use_cuda: bool):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (the slowest rank's time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------- clocks

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    """Samples the SM clock, its maximum and the clock-event reasons of one
    GPU from a background thread through NVML (read-only queries), falling
    back to `nvidia-smi --query-gpu ... -lms`."""

    def __init__(self, uuid: str | None, period_s: float = 0.002):
        self.uuid = uuid
        self.period = period_s
        self.samples = []  # (t, sm_mhz, reasons_mask, power_w)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thr = None
        self._proc = None
        self._nvml = None
        self._dev = None

    def _init_nvml(self) -> bool:
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        dev = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(dev)) == 0
        if not ok:
            ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(dev)) == 0
        if not ok:
            return False
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        self._nvml, self._dev = nv, dev
        self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return True

    def _loop_nvml(self):
        nv, dev = self._nvml, self._dev
        clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            t = time.perf_counter()
            if nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk)) == 0:
                r = rs.value if self._reason_fn(dev, ctypes.byref(rs)) == 0 else 0
                p = pw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(dev, ctypes.byref(pw)) == 0 else None
                self.samples.append((t, clk.value, r, p))
            time.sleep(self.period)

    def _loop_smi(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm = float(parts[1])
                self.max_mhz = float(parts[2])
                pw = float(parts[3])
                r = int(parts[4], 16) if parts[4].startswith("0x") else 0
            except ValueError:
                continue
            self.samples.append((time.perf_counter(), sm, r, pw))
            if self._stop.is_set():
                break

    def start(self):
        if self._init_nvml():
            self.source = "nvml"
            self._thr = threading.Thread(target=self._loop_nvml, daemon=True)
        else:
            self.source = "nvidia-smi"
            q = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"
            cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "20"]
            if self.uuid:
                cmd += ["-i", "GPU-" + self.uuid]
            try:
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                              text=True)
            except OSError:
                self.source = None
                return self
            self._thr = threading.Thread(target=self._loop_smi, daemon=True)
        self._thr.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 5.0:
            time.sleep(0.005)
        return self

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        if self._thr is not None:
            self._thr.join(timeout=2.0)

    def summary(self, t_begin: float, t_end: float):
        win = [s for s in self.samples if t_begin <= s[0] <= t_end]
        if not win:  # region shorter than the sampling period: nearest samples
            win = sorted(self.samples, key=lambda s: min(abs(s[0] - t_begin), abs(s[0] - t_end)))[:3]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.source}
        mask = 0
        for s in win:
            mask |= s[2]
        reasons = sorted(name for bit, name in _REASONS.items() if mask & bit and bit != 0x1)
        pw = [s[3] for s in win if s[3] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(win), "power_w_max": max(pw) if pw else None,
                "source": self.source}


# ----------------------------------------------------------------------------- helpers

def measured_peak():
    """MXFP8 dense peak: the measured BF16 burst GEMM rate x the nominal
    MXFP8/BF16 ratio; (value, source text)."""
    f = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(f.read_text())
        bf = float(d["bf16_tflops"])
        return bf * FP8_OVER_BF16, f"measured bf16 burst {bf} TFLOP/s x {FP8_OVER_BF16} (of measured)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_BURST * FP8_OVER_BF16, \
            f"fallback bf16 {FALLBACK_BF16_BURST} TFLOP/s x {FP8_OVER_BF16} (of fallback)"


def measured_hbm():
    """HBM copy bandwidth in GB/s; (value, source text)."""
    try:
        d = json.loads((ROOT / "MEASURED_PEAKS.json").read_text())
        v = float(d["hbm_gbs"])
        return v, f"measured copy {v} GB/s (of measured)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, f"fallback {FALLBACK_HBM_GBS} GB/s (of fallback)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary
    of this workload, if it was taken on the current kernel source; else
    None."""
    try:
        text = (PROFILES / f"mxgemm_kernel_{workload}.md").read_text()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, _, v = line.strip()[2:].partition(":")
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def oracle_rate_sample(prob, budget_s: float, max_rows: int | None = None):
    """Time the CPU oracle on whole output rows of `prob` for about budget_s
    seconds.  Returns (seconds, rows, threads)."""
    import numpy as np
    import oracle
    th = oracle.host_threads()
    t = time.perf_counter()
    oracle.rows(prob.A, prob.As, prob.B, prob.Bs, rows=np.arange(min(th, prob.M)), threads=th)
    dt = max(time.perf_counter() - t, 1e-6)
    per_row = dt / min(th, prob.M)
    rows = int(max(th, min(prob.M if max_rows is None else max_rows, budget_s / per_row)))
    rows = min(rows, prob.M)
    t = time.perf_counter()
    oracle.rows(prob.A, prob.As, prob.B, prob.Bs, rows=np.arange(rows), threads=th)
    return time.perf_counter() - t, rows, th


# ----------------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The CPU oracle as it stands, on the same workload; rank 0 only."""
    if rank != 0:
        return 0
    import numpy as np
    import mx_inputs
    import oracle
    prob = mx_inputs.WORKLOADS[args.workload]()
    M, N, K = prob.M, prob.N, prob.K
    th = oracle.host_threads()
    # rows per step so that warmup + steps take about args.ref_budget seconds
    t = time.perf_counter()
    oracle.rows(prob.A, prob.As, prob.B, prob.Bs, rows=np.arange(min(th, M)), threads=th)
    per_row = (time.perf_counter() - t) / min(th, M)
    rows = int(max(1, min(M, args.ref_budget / max(per_row, 1e-9) / (args.steps + args.warmup))))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.rows(prob.A, prob.As, prob.B, prob.Bs, rows=rng.integers(0, M, rows), threads=th)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.rows(prob.A, prob.As, prob.B, prob.Bs, rows=rng.integers(0, M, rows), threads=th)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K * args.steps
    value = flops / dt / 1e12
    sample = f"{rows} random output rows of {M} per step (all {N} columns, K={K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "out": prob.out_dtype,
                   "arm": "CPU FP64 oracle (plain definition), host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": th, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_quantize(args, world, rank, local):
    """The MX quantizer (mxgemm_quantize) on an R x C FP32 or BF16 matrix:
    HBM-bound, reported in GB/s of algorithmic traffic (read X, write codes
    and scales), checked bit for bit against the oracle on a row sample."""
    import numpy as np
    import torch
    import block_scaled_gemm_gb300 as mx
    from block_scaled_gemm_gb300 import _build
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the quantizer has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, True)
    _build.build()
    R, C = args.q_rows, args.q_cols
    dt = torch.bfloat16 if args.q_dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(0)
    x = (torch.randn((R, C), generator=g) * torch.exp(torch.randn((R, 1), generator=g) * 4)).to(dt)
    X = x.to(dev)
    cols = args.q_along == "cols"
    sr = args.q_round == "sr"
    # stochastic rounding reads one random 32-bit word per value (an input)
    rbits = (torch.randint(-2 ** 31, 2 ** 31, (R, C), generator=g, dtype=torch.int64)
             .to(torch.int32).to(dev) if sr else None)
    codes = torch.empty((R, C), dtype=torch.uint8, device=dev)
    scales = torch.empty((C, R // 32) if cols else (R, C // 32), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if not args.no_flush else None
    stream = torch.cuda.current_stream(dev)
    nbytes = R * C * x.element_size() + R * C + R * C // 32 + (R * C * 4 if sr else 0)
    for _ in range(args.warmup):
        mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=cols, stream=stream, rand_bits=rbits)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(None).start()
    torch.cuda.synchronize(dev)
    barrier(dist)
    t_begin = time.perf_counter()
    for a, b in ev:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=cols, stream=stream, rand_bits=rbits)
        b.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.perf_counter()
    sampler.stop()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dist, dev)
    gbs = nbytes * world * args.steps / (ms * 1e-3) / 1e9
    hbm, hbm_src = measured_hbm()
    parity = None
    if rank == 0:
        import oracle
        rb = rbits.cpu().numpy().view(np.uint32) if sr else None
        if cols:
            # a sample of whole columns (a column's blocks run down all R rows)
            cs = np.random.default_rng(1).integers(0, C, 64)
            rc, rs = oracle.quantize_e4m3(x[:, cs], along_cols=True,
                                          rand_bits=None if rb is None else rb[:, cs])
            parity = {"cols": int(cs.size),
                      "codes_equal": bool(np.array_equal(codes.cpu().numpy()[:, cs], rc)),
                      "scales_equal": bool(np.array_equal(scales.cpu().numpy()[cs], rs))}
        else:
            rows = np.random.default_rng(1).integers(0, R, 64)
            rc, rs = oracle.quantize_e4m3(x[rows], rand_bits=None if rb is None else rb[rows])
            parity = {"rows": int(rows.size),
                      "codes_equal": bool(np.array_equal(codes.cpu().numpy()[rows], rc)),
                      "scales_equal": bool(np.array_equal(scales.cpu().numpy()[rows], rs))}
        print(json.dumps({
            "metric": "MX quantizer GB/s (read X + write E4M3 codes + E8M0 scales"
                      + (" + read random words)" if sr else ")"),
            "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": args.q_dtype, "data": "synthetic",
            "config": {"workload": f"quantize_{R}x{C}_{args.q_dtype}_{args.q_along}"
                                   + ("_sr" if sr else ""), "R": R,
                       "C": C, "blocks": "32 down columns" if cols else "32 along rows",
                       "rounding": "stochastic" if sr else "nearest even",
                       "l2": "flushed between timed steps" if flush is not None else "not flushed"},
            "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / world / hbm, "peak_source": hbm_src,
                         "algorithmic_bytes": nbytes,
                         "kernel": "mx_quantize_cols_kernel" if cols else "mx_quantize_rows_kernel"},
            "gpu_launches": args.steps,
            "clocks": sampler.summary(t_begin, t_end),
            "parity": parity,
        }), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


class GemmSteps:
    """The calls of one step of a workload through the C interface (one
    mxgemm_run, or the chained use_acc calls of a K-split workload), with
    device operands prepared once."""

    def __init__(self, mx, h, prob, dev, packed: bool, stream, elems_packed: bool = False,
                 b_nk: bool = False):
        import torch
        import mx_inputs
        self.mx, self.h, self.prob, self.stream = mx, h, prob, stream
        self.out_code = mx.OUT_F32 if prob.out_dtype == "f32" else mx.OUT_BF16
        tdt = torch.float32 if prob.out_dtype == "f32" else torch.bfloat16
        self.C = torch.zeros((prob.M, prob.N), dtype=tdt, device=dev)
        self.calls = []
        chunks = [prob.chunk(c) for c in range(prob.k_chunks)] if prob.k_chunks > 1 else \
            [(prob.A, prob.As, prob.B, prob.Bs, prob.K)]
        self.keep = []
        for c, (A, As, B, Bs, K) in enumerate(chunks):
            if packed:
                As = mx_inputs.pack_scales(As)
                Bs = mx_inputs.pack_scales(Bs, along_cols=True)
            if b_nk:
                B = B.t().contiguous()  # B handed over as N x K (outside the step)
            if elems_packed:
                # 6- and 4-bit operands handed over in the tensor cores'
                # packed form (a host-side layout change, outside the step)
                fa, fb = prob.meta.get("formats", ("e4m3", "e4m3"))
                if mx_inputs.FORMAT_BITS[fa] < 8:
                    A = mx_inputs.pack_elements(A, mx_inputs.FORMAT_BITS[fa])
                if mx_inputs.FORMAT_BITS[fb] < 8:
                    B = mx_inputs.pack_elements(B, mx_inputs.FORMAT_BITS[fb])
            t = [x.to(dev) for x in (A, As, B, Bs)]
            self.keep.append(t)
            # a K-split workload accumulates every call into C (use_acc)
            ua = 1 if (prob.use_acc or c > 0) else 0
            self.calls.append((prob.M, prob.N, K, *t, self.C, ua, self.out_code))
        self.flops = 2.0 * prob.M * prob.N * prob.K

    def run(self, k_events=None):
        mx = self.mx
        for i, (M, N, K, A, As, B, Bs, C, ua, oc) in enumerate(self.calls):
            if k_events is not None:
                mx.mxgemm_set_profile_events(self.h, k_events[i][0], k_events[i][1])
            mx.mxgemm_run(self.h, M, N, K, A, As, B, Bs, C, ua, oc, self.stream)
        if k_events is not None:
            mx.mxgemm_set_profile_events(self.h, None, None)

    def alg_bytes(self) -> int:
        """Algorithmic HBM bytes of one step: operands, scales, C written
        (and read by every use_acc call)."""
        ob = 4 if self.prob.out_dtype == "f32" else 2
        total = 0
        for (M, N, K, *_rest, ua, _oc) in self.calls:
            total += M * K + K * N + (M + N) * K // 32 + M * N * ob * (2 if ua else 1)
        return total


def _events(torch, n):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    return ev


def _prime_events(torch, stream, evs):
    # torch creates the CUDA events lazily, at their first record
    for a, b in evs:
        a.record(stream)
        b.record(stream)


def time_workload(torch, ws: GemmSteps, steps: int, warmup: int, flush, dev):
    """Per-step CUDA-event times (ms) of `steps` steps with L2 flushed
    between steps (outside the events), per-step GEMM-kernel times (the
    library's events around each kernel launch, a second loop), and per-step
    times of back-to-back steps with no flush (hot L2)."""
    stream = ws.stream
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        ws.run()
    s_ev = _events(torch, steps)
    k_ev = [_events(torch, len(ws.calls)) for _ in range(steps)]
    h_ev = _events(torch, steps)
    _prime_events(torch, stream, s_ev + h_ev + [e for k in k_ev for e in k])
    torch.cuda.synchronize(dev)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        s_ev[i][0].record(stream)
        ws.run()
        s_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ws.run(k_events=k_ev[i])
    for i in range(steps):
        h_ev[i][0].record(stream)
        ws.run()
        h_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step = [a.elapsed_time(b) for a, b in s_ev]
    kern = [sum(a.elapsed_time(b) for a, b in k) for k in k_ev]
    hot = [a.elapsed_time(b) for a, b in h_ev]
    return step, kern, hot


def roofline_of(ws: GemmSteps, kern_ms: float, peak, peak_src, hbm, hbm_src):
    """Tensor-bound when the arithmetic intensity is above the ridge (peak
    FLOP/s / HBM bytes/s), else HBM-bound; achieved from the kernel time."""
    ab = ws.alg_bytes()
    if ws.flops / ab >= peak * 1e12 / (hbm * 1e9):
        a = ws.flops / (kern_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": a, "peak": peak, "unit": UNIT, "frac": a / peak,
                "peak_source": peak_src, "algorithmic_bytes": ab}
    gbs = ab / (kern_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "peak_source": hbm_src, "algorithmic_bytes": ab,
            "tflops": ws.flops / (kern_ms * 1e-3) / 1e12}


def spot_parity(torch, ws: GemmSteps, a_fmt, b_fmt, n=256, seed=1):
    """Run one fresh step (C zeroed first: a use_acc chain then holds exactly
    the product) and compare n seeded points with the oracle."""
    import numpy as np
    import oracle
    p = ws.prob
    ws.C.zero_()
    ws.run()
    torch.cuda.synchronize()
    g = np.random.default_rng(seed)
    I, J = g.integers(0, p.M, n), g.integers(0, p.N, n)
    ref, bound = oracle.points(p.A, p.As, p.B, p.Bs, I, J, a_fmt=a_fmt, b_fmt=b_fmt)
    got = ws.C.float().cpu().numpy()[I, J]
    acc = oracle.accept(got, ref, bound, "f32" if p.out_dtype == "f32" else "bf16")
    return {"points": int(I.size), "ok": acc["ok"], "max_err_over_bound": acc["max_err_over_bound"]}


def run_mx(args, world, rank, local):
    import numpy as np
    import torch

    import block_scaled_gemm_gb300 as mx
    import mx_inputs
    from block_scaled_gemm_gb300 import _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GEMM has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, True)
    _build.build()

    prob = mx_inputs.WORKLOADS[args.workload]()
    if (args.a_format, args.b_format) != ("e4m3", "e4m3"):
        prob = mx_inputs.with_formats(prob, args.a_format, args.b_format)
    M, N, K = prob.M, prob.N, prob.K
    packed = args.scale_layout == "packed"
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev) if not args.no_flush else None
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = measured_peak()
    hbm, hbm_src = measured_hbm()

    h = mx.mxgemm_create(local)
    if args.mode is not None:
        mx.mxgemm_set_option(h, mx.OPT_MODE, args.mode)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, FORMATS.index(args.a_format))
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FORMATS.index(args.b_format))
    elems_packed = args.element_layout == "packed"
    if elems_packed:
        mx.mxgemm_set_option(h, mx.OPT_ELEMENT_LAYOUT, mx.ELEMS_PACKED)
    b_nk = args.b_major == "nk"
    if b_nk:
        mx.mxgemm_set_option(h, mx.OPT_B_MAJOR, mx.B_N_BY_K)
    if packed:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_PACKED)
    ws = GemmSteps(mx, h, prob, dev, packed, stream, elems_packed, b_nk)
    flops = ws.flops

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        ws.run()
    torch.cuda.synchronize(dev)
    st, det = mx.mxgemm_get_device_status(h)
    if st != 0:
        raise SystemExit(f"device status {st} detail {det:#x}")

    s_ev = _events(torch, args.steps)
    k_ev = [_events(torch, len(ws.calls)) for _ in range(args.steps)]
    h_ev = _events(torch, args.steps)
    _prime_events(torch, stream, s_ev + h_ev + [e for k in k_ev for e in k])
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    launches0 = mx.mxgemm_get_launch_count(h)

    # ---- the timed region: exactly args.steps steps, L2 flushed between them
    barrier(dist)
    torch.cuda.synchronize(dev)
    t_begin = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        s_ev[i][0].record(stream)
        ws.run()
        s_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t_end = time.perf_counter()
    launches = mx.mxgemm_get_launch_count(h) - launches0
    st, det = mx.mxgemm_get_device_status(h)
    if st != 0:
        raise SystemExit(f"device status {st} detail {det:#x}")
    clocks = sampler.summary(t_begin, t_end)

    # the GEMM kernel alone, for its roofline: the library records events
    # around each kernel launch (a second loop, so that events between a
    # prepass and the kernel do not disturb the timed steps above); then the
    # same steps back to back with no flush (hot L2)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ws.run(k_events=k_ev[i])
    for i in range(args.steps):
        h_ev[i][0].record(stream)
        ws.run()
        h_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)

    step_list = [a.elapsed_time(b) for a, b in s_ev]
    kern_list = [sum(a.elapsed_time(b) for a, b in k) for k in k_ev]
    hot_list = [a.elapsed_time(b) for a, b in h_ev]
    step_ms_max = max_over_ranks(sum(step_list), dist, dev)
    value = flops * world * args.steps / (step_ms_max * 1e-3) / 1e12
    kern_avg_ms = sum(kern_list) / len(kern_list)

    # ---- sustained: the same step back to back for a few seconds (the
    # power-capped rate of a long run; also what a clock sampler needs)
    sustained = None
    if args.sustain_s > 0:
        per = max(statistics.median(hot_list), 1e-3)
        n_sus = int(max(args.steps, min(200000, args.sustain_s * 1e3 / per)))
        e0, e1 = _events(torch, 1)[0]
        torch.cuda.synchronize(dev)
        ts0 = time.perf_counter()
        e0.record(stream)
        for _ in range(n_sus):
            ws.run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts1 = time.perf_counter()
        sus_ms = e0.elapsed_time(e1)
        sustained = {"steps": n_sus, "seconds": sus_ms * 1e-3, "l2": "not flushed (back to back)",
                     "value": flops * n_sus / (sus_ms * 1e-3) / 1e12, "unit": UNIT,
                     "frac_of_peak": flops * n_sus / (sus_ms * 1e-3) / 1e12 / peak,
                     "clocks": sampler.summary(ts0, ts1)}
        st, det = mx.mxgemm_get_device_status(h)
        if st != 0:
            raise SystemExit(f"device status {st} detail {det:#x}")

    # ---- the other workloads: step, kernel and hot-L2 medians, roofline,
    # spot parity (each workload's own inputs, generated here)
    table = None
    if args.workloads != "none" and rank == 0:
        table = {}
        names = [n for n in WORKLOAD_TABLE if n != args.workload]
        for name in names:
            pw = mx_inputs.WORKLOADS[name]()
            hw = mx.mxgemm_create(local)
            try:
                wsw = GemmSteps(mx, hw, pw, dev, packed, stream)
                n_steps = max(args.steps, 50) if pw.M * pw.N * pw.K <= (1 << 36) else args.steps
                step_w, kern_w, hot_w = time_workload(torch, wsw, n_steps, max(args.warmup, 5),
                                                      flush, dev)
                st, det = mx.mxgemm_get_device_status(hw)
                km = statistics.median(kern_w)
                row = {"M": pw.M, "N": pw.N, "K": pw.K, "calls_per_step": len(wsw.calls),
                       "out": pw.out_dtype, "steps": n_steps,
                       "step_us_median": statistics.median(step_w) * 1e3,
                       "kernel_us_median": km * 1e3,
                       "hot_l2_step_us_median": statistics.median(hot_w) * 1e3,
                       "tflops_step": wsw.flops / (statistics.median(step_w) * 1e-3) / 1e12,
                       "roofline": roofline_of(wsw, km, peak, peak_src, hbm, hbm_src),
                       "status": st}
                if not args.no_cpu:
                    row["parity"] = spot_parity(torch, wsw, args.a_format, args.b_format)
                table[name] = row
                del wsw
            finally:
                mx.mxgemm_destroy(hw)
            del pw
            torch.cuda.empty_cache()

    # spot parity of the headline result against the oracle (rank 0)
    parity = None
    if rank == 0 and not args.no_cpu:
        parity = spot_parity(torch, ws, args.a_format, args.b_format)

    # ---- end to end through the C interface: pinned host operands in, C out
    e2e = None
    if args.e2e_steps > 0:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        sA = mx_inputs.pack_scales(prob.As) if packed else prob.As
        sB = mx_inputs.pack_scales(prob.Bs, along_cols=True) if packed else prob.Bs
        eA, eB = prob.A, (prob.B.t().contiguous() if b_nk else prob.B)
        if elems_packed:
            if mx_inputs.FORMAT_BITS[args.a_format] < 8:
                eA = mx_inputs.pack_elements(eA, mx_inputs.FORMAT_BITS[args.a_format])
            if mx_inputs.FORMAT_BITS[args.b_format] < 8:
                eB = mx_inputs.pack_elements(eB, mx_inputs.FORMAT_BITS[args.b_format])
        hA, hAs, hB, hBs = (t.contiguous().pin_memory() for t in (eA, sA, eB, sB))
        hC = torch.empty((M, N), dtype=ws.C.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hA, hAs, hB, hBs))
        d2h = hC.numel() * hC.element_size()
        ua0 = 1 if prob.use_acc else 0
        # the host-buffer entry point: B in, then A rows in / C rows out in
        # slabs overlapped with the slabs' GEMMs; the copies are in the
        # timed region of every step (one call over the whole K)
        def e2e_step():
            mx.mxgemm_run_host(h, M, N, K, hA, hAs, hB, hBs, hC, ua0, ws.out_code, stream)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(dist)
        e0, e1 = _events(torch, 1)[0]
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        if prob.use_acc:
            h2d += hC.numel() * hC.element_size()  # use_acc: C is copied in as well
        e2e = {"value": flops * world * e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "entry_point": "mxgemm_run_host"}
        del hA, hAs, hB, hBs, hC
    mx.mxgemm_destroy(h)
    sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu:
        dt, rows, th = oracle_rate_sample(prob, args.cpu_budget)
        cpu = {"value": 2.0 * rows * N * K / dt / 1e12, "unit": UNIT, "cores": th, "kind": "oracle",
               "sample": f"first {rows} of {M} output rows (all {N} columns, K={K}), {dt:.1f} s"}

    if rank == 0:
        roofline = roofline_of(ws, kern_avg_ms, peak, peak_src, hbm, hbm_src)
        roofline.update({"traffic": profiled_traffic(args.workload), "kernel": "mxgemm_kernel",
                         "kernel_avg_us": kern_avg_ms * 1e3})
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8",
            "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                       "a": f"{args.a_format.upper()} M x K (K-major), scales E8M0 per 32 K",
                       "b": f"{args.b_format.upper()} K x N (N-major), scales E8M0 per 32 K",
                       "out": prob.out_dtype, "use_acc": int(prob.use_acc),
                       "calls_per_step": len(ws.calls), "accumulate": "fp32",
                       "l2": ("flushed between timed steps (write of 2x L2, outside the events)"
                              if flush is not None else "not flushed"),
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "tile_mode": args.mode if args.mode is not None else "auto",
                       "a_format": args.a_format, "b_format": args.b_format,
                       "scale_layout": args.scale_layout, "element_layout": args.element_layout,
                       "b_major": args.b_major},
            "timing": {"step_us_median": statistics.median(step_list) * 1e3,
                       "step_us_mean": sum(step_list) / len(step_list) * 1e3,
                       "kernel_us_median": statistics.median(kern_list) * 1e3,
                       "kernel_us_mean": kern_avg_ms * 1e3,
                       "hot_l2_step_us_median": statistics.median(hot_list) * 1e3,
                       "tflops_step_median": flops / (statistics.median(step_list) * 1e-3) / 1e12,
                       "tflops_hot_l2_median": flops / (statistics.median(hot_list) * 1e-3) / 1e12},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "sustained": sustained,
            "workloads": table,
            "parity": parity,
            "kernel_source_sha": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mx", "reference"], default="mx")
    import mx_inputs
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(mx_inputs.WORKLOADS))
    ap.add_argument("--mode", type=int, default=None, help="tile mode: 1 = 1-CTA, 2 = CTA pair")
    ap.add_argument("--op", default="gemm", choices=["gemm", "quantize"],
                    help="gemm (the headline) or the MX quantizer")
    ap.add_argument("--q-rows", type=int, default=8192)
    ap.add_argument("--q-cols", type=int, default=8192)
    ap.add_argument("--q-dtype", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--q-along", default="rows", choices=["rows", "cols"],
                    help="quantizer blocks: 32 along rows (A) or down columns (B)")
    ap.add_argument("--q-round", default="rn", choices=["rn", "sr"],
                    help="quantizer rounding: nearest even, or stochastic with one random word per value")
    ap.add_argument("--a-format", default="e4m3", choices=FORMATS)
    ap.add_argument("--b-format", default="e4m3", choices=FORMATS)
    ap.add_argument("--scale-layout", default="row-major", choices=["row-major", "packed"],
                    help="scales row-major (the workload's form; the run repacks them) or "
                         "pre-packed in the tensor cores' order (as mxgemm_quantize_ex writes them)")
    ap.add_argument("--element-layout", default="byte", choices=["byte", "packed"],
                    help="6- and 4-bit operands one code per byte (packed by the library each "
                         "call) or already in the tensor cores' packed form")
    ap.add_argument("--b-major", default="kn", choices=["kn", "nk"],
                    help="B handed over K x N (N contiguous, the default) or N x K (K contiguous, "
                         "a linear layer's weight)")
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline and spot parity")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workloads", default="all", choices=["all", "none"],
                    help="also measure the other workloads (the 'workloads' object)")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps for the sustained rate (0: skip)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds of oracle work for --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.op == "quantize":
        return run_quantize(args, world, rank, local)
    return run_mx(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
