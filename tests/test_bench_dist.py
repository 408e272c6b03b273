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
