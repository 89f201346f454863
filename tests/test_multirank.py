"""bench.py's multi-rank plumbing on CPU: two gloo ranks on 127.0.0.1 run the barrier,
the max over ranks and the weak-scaling aggregation that bench.py uses for N GPUs."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each rank's timed region differs; the job's time is the slowest rank's
    seconds = bench.max_over_ranks(1.0 + 0.5 * rank, w)
    rate = bench.weak_scaling_rate(100, 10, w, seconds)
    results[rank] = (seconds, rate)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_rate():
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time, and the rate counts both ranks' units
    for rank in range(world):
        seconds, rate = results[rank]
        assert seconds == pytest.approx(1.5)
        assert rate == pytest.approx(100 * 10 * world / 1.5)


def test_reference_arm_rank_nonzero_does_no_work():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps = 1
        warmup = 0
    assert bench.run_reference(A(), 1, 2) is None
