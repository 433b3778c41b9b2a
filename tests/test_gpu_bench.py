"""The benchmark's JSON line on a GB300: a short run of `bench.py` on a small
workload must print one line with the measurement contract's keys, a
roofline of the GEMM kernel, an oracle baseline, an end-to-end figure with
its host copies counted, a launch count from the library and the clocks of
the timed region; and its spot parity against the oracle must hold."""
import json
import os
import subprocess
import sys
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parents[1]


def _run(*args):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=str(ROOT), env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_gemm_line_keeps_the_contract():
    d = _run("--workload", "square_256", "--steps", "5", "--warmup", "3", "--workloads", "none",
             "--sustain-s", "0.2", "--e2e-steps", "3", "--cpu-budget", "0.5")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["steps"] == 5 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "square_256"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    r = d["roofline"]
    assert r["bound"] in ("tensor", "hbm") and r["unit"] in ("TFLOP/s", "GB/s")
    assert r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    # every step copies A, B and their scales in and C out
    M = N = K = 256
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] >= M * K + K * N + (M + N) * K // 32
    assert e["d2h_bytes_per_step"] >= M * N * 4
    assert d["gpu_launches"] >= d["steps"]  # at least one library kernel per step
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    assert not d.get("workloads")  # --workloads none
    assert d["parity"]["ok"] and d["parity"]["points"] > 0


def test_skinny_line_reports_hbm():
    d = _run("--workload", "skinny_16x8192x8192", "--steps", "5", "--warmup", "3", "--workloads", "none",
             "--sustain-s", "0.2", "--e2e-steps", "2", "--cpu-budget", "0.5")
    assert d["config"]["workload"] == "skinny_16x8192x8192"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
