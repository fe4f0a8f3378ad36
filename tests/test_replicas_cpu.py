"""The N > 1 path of bench.py without a GPU: two gloo ranks on the host.

bench.py runs one replica of the whole head per GPU (the path has no
exchange step here), takes the slowest rank's times with an all-reduce MAX
and reports the bytes of all replicas over that time.  These tests run the
same reduction and throughput arithmetic under a gloo process group of two
ranks, rendezvous on 127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r was slower on the first timing and faster on the second
        local = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        red = bench.aggregate_over_ranks(local, world)
        gbs = bench.job_throughput_gbs(bench.step_bytes(), 10, world, red[0])
        q.put((rank, red, gbs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    for rank, red, gbs in out:
        assert red == [2.0, 5.0, 0.5]                  # element-wise max over the ranks
        assert gbs == pytest.approx(bench.step_bytes() * 10 * world / 2.0 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_throughput_gbs(1_000_000_000, 2, 1, 2.0) == pytest.approx(1.0)
