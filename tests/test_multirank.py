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


RANK_SCRIPT = """
import json, os, sys
sys.path.insert(0, {root!r})
import bench
r, w, local = bench.dist_init()
bench.barrier(w)
t = bench.max_over_ranks(1.0 + r, w)
with open(os.path.join({out!r}, "rank%d.json" % r), "w") as f:
    json.dump([r, w, local, t], f)
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_bench_starts_its_own_ranks(tmp_path):
    """``bench.py --gpus N`` outside torchrun starts N ranks through torchrun's launcher;
    the command it builds runs two gloo ranks here that rendezvous on 127.0.0.1."""
    import subprocess
    sys.path.insert(0, ROOT)
    import bench
    script = tmp_path / "rank.py"
    script.write_text(RANK_SCRIPT.format(root=ROOT, out=str(tmp_path)))
    cmd = bench.torchrun_command(2, _free_port(), str(script), [])
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, env=env, timeout=180, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    got = sorted(json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2))
    assert got == [[0, 2, 0, 2.0], [1, 2, 1, 2.0]]
