"""The bench's N > 1 logic on CPU: two gloo ranks agree on the slowest
rank's time, the whole-job value counts every rank's bytes, and the
reference arm does its work on rank 0 only."""
import os
import socket
import sys
import tempfile

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(torch, dist, 1.0 + 0.5 * rank, "cpu")
        v = bench.whole_job_gbs(1e9, 10, t, world)
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(f"{t} {v}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank, args=(world, _free_port(), d), nprocs=world, start_method="spawn")
        got = [open(os.path.join(d, f"r{r}")).read().split() for r in range(world)]
    for t, v in got:
        assert float(t) == 1.5                                   # rank 1 was slower
        assert abs(float(v) - world * 1e9 * 10 / 1.5 / 1e9) < 1e-9  # both ranks' bytes over that time


def test_without_a_process_group_the_local_time_stands():
    import bench
    assert bench.max_over_ranks(torch, None, 2.5, "cpu") == 2.5
    assert bench.whole_job_gbs(4e9, 2, 1.0, 1) == 8.0


def test_reference_arm_other_ranks_do_no_work():
    import bench

    class A:
        steps, warmup = 1, 1
    assert bench.reference_arm(A, rank=1, world=2) == 0
