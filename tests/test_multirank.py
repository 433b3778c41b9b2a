"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2): each rank
reports a different time, every rank must see the slowest one, and the
reference arm runs on rank 0 only.  No GPU is involved: under torchrun the
path runs independent replicas, one per GPU, with no collective on the data
path; these helpers are the only cross-rank steps."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, use_cuda=False)
    bench.barrier(dist)
    mine = 10.0 + 5.0 * r          # rank r's time
    slowest = bench.max_over_ranks(mine, dist, "cpu")
    bench.barrier(dist)
    Path(out_dir, f"rank{r}.txt").write_text(f"{w} {r} {slowest}")
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    got = sorted(Path(tmp_path).glob("rank*.txt"))
    assert len(got) == world
    for f in got:
        w, r, slowest = f.read_text().split()
        assert int(w) == world
        assert float(slowest) == 15.0   # every rank sees the slowest rank's time


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    class Args:
        workload = "square_256"
        steps = 3
        warmup = 3
        ref_budget = 0.5

    assert bench.run_reference(Args(), 2, 1) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1, use_cuda=False) is None
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    bench.barrier(None)


def test_reference_arm_line_keeps_the_contract(capsys):
    # rank 0 of one: one JSON line with the keys the measurement contract
    # names, the CPU baseline describing this run and no host copies
    import json
    import bench

    class Args:
        workload = "square_256"
        steps = 3
        warmup = 3
        ref_budget = 0.5

    assert bench.run_reference(Args(), 1, 0) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "square_256"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
