"""The benchmark's multi-rank helpers on the CPU: two `gloo` ranks set up
from the environment the launcher provides, meet at the barrier, and agree on
the maximum of their step times (the time the job is charged with)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, wsz, local = bench.dist_setup()
    assert (r, wsz, local) == (rank, world, rank)
    bench.barrier(wsz)
    slowest = bench.max_over_ranks(1.5 + rank, wsz)  # rank 1 is the slower one
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(world)]
    assert got == [2.5, 2.5]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)  # no-op without a process group
