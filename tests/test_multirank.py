"""Multi-rank host logic of bench.py under gloo on CPU (world size 2): the
job time is the slowest rank's, the job value counts every rank's units, and
only rank 0 of the reference arm prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = 10.0 + 5.0 * rank                      # rank 1 is slower
        slowest = bench.max_over_ranks(mine)
        value = bench.job_throughput(world, 100, 1000, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 100 * 1000 / 0.015)


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(1, 10, 50, 1.0) == pytest.approx(10 * 50 / 1e-3)
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_prints_on_rank_0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload = "1"
        steps = 1
        warmup = 0
        ref_budget_s = 0.5
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args, 1, 2)               # rank 1 of 2: no work, no output
    assert buf.getvalue() == ""
    with redirect_stdout(buf):
        bench.run_reference(Args, 0, 1)
    import json
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["warmup"] >= 3
