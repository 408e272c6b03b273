"""The multi-process timing plumbing of bench.py on CPU ranks (gloo, world size 2).

Rows are independent, so several GPUs only split the batch (weak scaling):
the one cross-rank step is the timing, a barrier and the slowest rank's time.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r "took" 1 + r seconds: the slowest rank's time is reported
        t = bench.max_over_ranks(1.0 + rank, world)
        rows = bench.aggregate_rows_per_s(64, world, t)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{t} {rows}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    vals = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for t, rows in vals:
        assert float(t) == pytest.approx(2.0)
        assert float(rows) == pytest.approx(64 * world / 2.0)


def test_single_rank_helpers_are_identities():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)  # no process group needed
    assert bench.aggregate_rows_per_s(64, 1, 0.5) == pytest.approx(128.0)


def _bench(args, env_extra=None):
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], cwd=root, env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    import json

    from workloads import WORKLOADS

    import bench

    p = _bench(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == WORKLOADS[bench.HEADLINE].name
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0


def test_reference_arm_runs_on_rank_zero_only():
    p = _bench(["--impl", "reference", "--steps", "3", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_fewer_than_three_warmup_steps_are_refused():
    p = _bench(["--impl", "reference", "--steps", "3", "--warmup", "2"])
    assert p.returncode != 0
    assert "warmup" in p.stderr
