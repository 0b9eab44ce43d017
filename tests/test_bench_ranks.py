"""The multi-rank path of bench.py on CPU: two gloo ranks (no GPU needed).

With N GPUs the bench runs one independent replica per rank (the path has no
data exchange between replicas); rank 0 reports the whole job's bytes over the
slowest rank's time.  These tests run the rank aggregation over gloo with
world size 2, and check that the reference arm prints only on rank 0.
"""

import io
import os
import socket
import sys
import contextlib

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(times[rank], world)
    value = bench.whole_job_gbs(1_000_000_000, 10, slowest, world)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    times = [12.5, 20.0]          # rank 1 is slower
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 20.0
        # 2 ranks x 1 GB x 10 steps over 20 ms
        assert value == pytest.approx(2 * 1e9 * 10 / 0.020 / 1e9)


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_gbs(2e9, 4, 8.0, 1) == pytest.approx(1000.0)


def test_reference_arm_prints_only_on_rank_0(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=0, gpus=2, cpu_workers=1))()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
