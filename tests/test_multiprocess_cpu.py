"""The multi-rank path of the benchmark on CPU (gloo, world size 2, 127.0.0.1): every rank runs
its own batch (weak scaling, no data-path collective); the step time is the slowest rank's,
taken after a barrier; only rank 0 runs the reference arm."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = 1.0 + 2.0 * rank  # rank 1 is the slower one
    bench.barrier(world)
    slowest = bench.reduce_max(torch, world, ms, device="cpu")
    q.put((rank, slowest, bench.job_value(world, 4096, slowest)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_step_and_the_whole_job():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in out) == [0, 1]
    for _, slowest, value in out:
        assert slowest == 3.0
        assert value == pytest.approx(2 * 4096 / 3e-3)


def test_reference_arm_runs_on_rank_0_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(Args, 1)
    assert buf.getvalue() == ""
