"""The bench's multi-GPU mode is replicas only: every rank runs its own stack and
the job's value is all ranks' units over the slowest rank's time.  Its host-side
plumbing (rank environment, barrier, max over ranks) checked with two gloo
ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        # per-rank times differ; every rank must report the slowest
        slowest = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
        units = 100 * (rank + 1)          # each rank's own work
        total = torch.tensor([units], dtype=torch.float64)
        dist.all_reduce(total)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%d %d %d %r %r\n" % (w, r, local, slowest, total.item() / slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    rows = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for r, row in enumerate(rows):
        w, rank, local, slowest, value = int(row[0]), int(row[1]), int(row[2]), float(row[3]), \
            float(row[4])
        assert (w, rank, local) == (world, r, r)
        assert slowest == 11.0                      # max over ranks, the same on every rank
        assert value == pytest.approx(300 / 11.0)   # all ranks' units over the slowest time


def test_single_process_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    bench.barrier(1)                                 # no process group needed
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
