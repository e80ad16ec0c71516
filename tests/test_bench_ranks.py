"""The multi-GPU host logic of bench.py on CPU: two gloo ranks, each with its own
replica's timings.  The path shards into independent replicas (one per GPU, no
data-path exchange), so what N > 1 adds is the max over ranks of the timings
and the whole-job aggregate; both are checked here without a GPU."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1), 7.0, 3.0 + 2 * rank]
        got = bench.max_over_ranks(mine, world, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(",".join(repr(x) for x in got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    want = [2.0, 5.0, 0.5, 7.0, 5.0]
    for r in range(world):
        got = [float(x) for x in (tmp_path / f"r{r}.txt").read_text().split(",")]
        assert got == want, (r, got)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_gbs(1, 446.9e6, 0.122)
    assert abs(one - 3663.1) < 0.1
    # two replicas, each the same bytes, the slower one's time
    assert abs(bench.job_gbs(2, 446.9e6, 0.122) - 2 * one) < 1e-6
