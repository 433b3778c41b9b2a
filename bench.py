#!/usr/bin/env python3
"""Benchmark of the GB300 MX block-scaled FP8 GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mx|reference]

One step = one C = A.B call through the C interface (scale repack prepasses +
the tcgen05 GEMM kernel) on the square 4096 x 4096 x 4096 MXFP8 workload
(E4M3 operands quantized per 32-element K block from N(0,1), E8M0 scale bytes
replaced by uniform integers in [123, 131], FP32 output), inputs resident in
HBM.  The operands plus C (97 MB) fit in the 126 MB L2, so a 256 MiB buffer
is written between timed steps (L2 flushed) and each step is timed with its
own CUDA events on the launching stream; the flush is outside the events.

Prints one JSON line: metric TFLOP/s = 2MNK / t (whole job), the roofline of
the GEMM kernel (timed alone by events the library records around its
launch) against the MXFP8 tensor peak, end-to-end TFLOP/s through the C
interface with pinned host buffers (H2D of A, B and scales + D2H of C inside
the timed region), SM clocks sampled during the timed region, and the CPU
oracle timed on a bounded sample of the same workload.

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
WORKLOAD = "square_4096"
FP8_OVER_BF16 = 2.0  # nominal dense MXFP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
FALLBACK_BF16_BURST = 1900.0  # TFLOP/s, used only when MEASURED_PEAKS.json is absent
FORMATS = ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"]  # C interface order (mxgemm_format_t)
FALLBACK_HBM_GBS = 6800.0     # GB/s, used only when MEASURED_PEAKS.json is absent
KERNEL_SOURCES = ["block_scaled_gemm_gb300/csrc/mxgemm_kernel.cuh",
                  "block_scaled_gemm_gb300/csrc/ptx.cuh"]
PROFILE_SUMMARY = ROOT / "profiles" / "mxgemm_kernel_square_4096.md"


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


def profiled_traffic():
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    try:
        text = PROFILE_SUMMARY.read_text()
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
    out_code = mx.OUT_F32 if prob.out_dtype == "f32" else mx.OUT_BF16
    tdt = torch.float32 if prob.out_dtype == "f32" else torch.bfloat16
    flops = 2.0 * M * N * K

    # scales as the run takes them: row-major (the default), or already in
    # the packed order the tensor cores read (no repack prepass)
    packed = args.scale_layout == "packed"
    sA = mx_inputs.pack_scales(prob.As) if packed else prob.As
    sB = mx_inputs.pack_scales(prob.Bs, along_cols=True) if packed else prob.Bs
    A, As, B, Bs = (t.to(dev) for t in (prob.A, sA, prob.B, sB))
    C = torch.empty((M, N), dtype=tdt, device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev) if not args.no_flush else None
    stream = torch.cuda.current_stream(dev)

    h = mx.mxgemm_create(local)
    if args.mode is not None:
        mx.mxgemm_set_option(h, mx.OPT_MODE, args.mode)
    mx.mxgemm_set_option(h, mx.OPT_A_FORMAT, FORMATS.index(args.a_format))
    mx.mxgemm_set_option(h, mx.OPT_B_FORMAT, FORMATS.index(args.b_format))
    if packed:
        mx.mxgemm_set_option(h, mx.OPT_SCALE_LAYOUT, mx.SCALES_PACKED)

    def step():
        if flush is not None:
            flush.zero_()
        mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, out_code, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, det = mx.mxgemm_get_device_status(h)
    if st != 0:
        raise SystemExit(f"device status {st} detail {det:#x}")

    mk = lambda: torch.cuda.Event(enable_timing=True)
    s_ev = [(mk(), mk()) for _ in range(args.steps)]
    k_ev = [(mk(), mk()) for _ in range(args.steps)]
    for a, b in s_ev + k_ev:  # create the CUDA events (torch creates them lazily)
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    launches0 = mx.mxgemm_get_launch_count(h)

    barrier(dist)
    torch.cuda.synchronize(dev)
    t_begin = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        s_ev[i][0].record(stream)
        mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, out_code, stream)
        s_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t_end = time.perf_counter()
    launches = mx.mxgemm_get_launch_count(h) - launches0
    sampler.stop()
    st, det = mx.mxgemm_get_device_status(h)
    if st != 0:
        raise SystemExit(f"device status {st} detail {det:#x}")

    # the GEMM kernel alone, for its roofline: the library records events
    # around the kernel launch (a second loop, so that the events between the
    # prepass and the kernel do not disturb the timed steps above)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        mx.mxgemm_set_profile_events(h, k_ev[i][0], k_ev[i][1])
        mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, out_code, stream)
    torch.cuda.synchronize(dev)
    mx.mxgemm_set_profile_events(h, None, None)

    step_ms = sum(a.elapsed_time(b) for a, b in s_ev)
    kern_ms = sum(a.elapsed_time(b) for a, b in k_ev)
    step_ms_max = max_over_ranks(step_ms, dist, dev)
    value = flops * world * args.steps / (step_ms_max * 1e-3) / 1e12
    kern_avg_ms = kern_ms / args.steps
    achieved = flops / (kern_avg_ms * 1e-3) / 1e12
    peak, peak_src = measured_peak()
    clocks = sampler.summary(t_begin, t_end)

    # spot parity of the timed result against the oracle (rank 0)
    parity = None
    if rank == 0 and not args.no_cpu:
        import oracle
        g = np.random.default_rng(1)
        I, J = g.integers(0, M, 256), g.integers(0, N, 256)
        ref, bound = oracle.points(prob.A, prob.As, prob.B, prob.Bs, I, J,
                                   a_fmt=args.a_format, b_fmt=args.b_format)
        got = C.float().cpu().numpy()[I, J]
        acc = oracle.accept(got, ref, bound, "f32" if prob.out_dtype == "f32" else "bf16")
        parity = {"points": int(I.size), "ok": acc["ok"],
                  "max_err_over_bound": acc["max_err_over_bound"]}

    # end to end through the C interface: pinned host operands in, C out
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    hA, hAs, hB, hBs = (t.contiguous().pin_memory() for t in (prob.A, sA, prob.B, sB))
    hC = torch.empty((M, N), dtype=tdt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hA, hAs, hB, hBs))
    d2h = hC.numel() * hC.element_size()

    # the host-buffer entry point: B in, then A rows in / C rows out in
    # slabs overlapped with the slabs' GEMMs; the copies are in the timed
    # region of every step
    def e2e_step():
        mx.mxgemm_run_host(h, M, N, K, hA, hAs, hB, hBs, hC, 0, out_code, stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(dist)
    e0, e1 = mk(), mk()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = flops * world * e2e_steps / (e2e_ms * 1e-3) / 1e12
    mx.mxgemm_destroy(h)

    cpu = None
    if rank == 0 and not args.no_cpu:
        dt, rows, th = oracle_rate_sample(prob, args.cpu_budget)
        cpu = {"value": 2.0 * rows * N * K / dt / 1e12, "unit": UNIT, "cores": th, "kind": "oracle",
               "sample": f"first {rows} of {M} output rows (all {N} columns, K={K}), {dt:.1f} s"}

    if rank == 0:
        # Tensor-bound when the arithmetic intensity is above the ridge
        # (peak FLOP/s / HBM bytes/s), else HBM-bound: achieved = algorithmic
        # bytes per launch / kernel time.
        alg_bytes = M * K + K * N + (M + N) * K // 32 + M * N * (4 if prob.out_dtype == "f32" else 2)
        hbm, hbm_src = measured_hbm()
        if 2.0 * M * N * K / alg_bytes >= peak * 1e12 / (hbm * 1e9):
            roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                        "frac": achieved / peak, "peak_source": peak_src}
        else:
            gbs = alg_bytes / (kern_avg_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                        "frac": gbs / hbm, "peak_source": hbm_src}
        roofline.update({"traffic": profiled_traffic() if args.workload == WORKLOAD else None,
                         "algorithmic_bytes": alg_bytes, "kernel": "mxgemm_kernel",
                         "kernel_avg_us": kern_avg_ms * 1e3})
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8",
            "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                       "a": f"{args.a_format.upper()} M x K (K-major), scales E8M0 per 32 K",
                       "b": f"{args.b_format.upper()} K x N (N-major), scales E8M0 per 32 K",
                       "out": prob.out_dtype, "use_acc": 0, "accumulate": "fp32",
                       "l2": ("flushed between timed steps (256 MiB write, outside the events)"
                              if flush is not None else "not flushed"),
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "tile_mode": args.mode if args.mode is not None else "auto",
                       "a_format": args.a_format, "b_format": args.b_format,
                       "scale_layout": args.scale_layout},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": launches,
            "clocks": clocks,
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
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline and spot parity")
    ap.add_argument("--e2e-steps", type=int, default=20)
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
