"""The multi-GPU path of bench.py on CPU: replicas over a world-size-2 gloo
process group.  The path has no data exchange; what the ranks share is the
timing rule (every per-rank time becomes the slowest rank's) and the
whole-job rate (world x per-replica bytes / slowest time).  The reference
arm runs on rank 0 only; other ranks return without work or output."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r measured (1 + r) ms per step and (10 - r) ms per decode
        got = bench.slowest_over_ranks([1.0 + rank, 10.0 - rank], dist, torch.device("cpu"))
        rate = bench.job_throughput(world, 1000, got[0] * 1e-3)
        q.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=90) for _ in range(world)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, got, rate in out:
        assert got == [2.0, 10.0], (rank, got)      # max over ranks of each time
        assert rate == pytest.approx(2 * 1000 / 2e-3)  # both replicas' bytes, slowest step


def test_single_process_is_identity():
    import torch

    import bench
    assert bench.slowest_over_ranks([3.0, 4.0], None, torch.device("cpu")) == [3.0, 4.0]
    assert bench.job_throughput(1, 500, 0.5) == 1000


def test_reference_arm_other_ranks_do_no_work(capsys):
    import bench
    ns = type("Args", (), {"steps": 1, "warmup": 1, "gpus": 2})()
    assert bench.run_reference(ns, 1, 2) is None
    assert capsys.readouterr().out == ""
