"""The N > 1 host logic of ``bench.py`` on CPU: two ``gloo`` ranks, each a
replica of the workload.  The slowest rank's times are what rank 0 reports,
the whole-job rate counts every replica's work, and the reference arm runs
on rank 0 only.  No GPU and no data-path collective are involved.
"""

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


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r's replica took (1 + r) ms per step, (2 + r) ms for the decode
        got = bench.max_over_ranks([1.0 + rank, 2.0 + rank, 10.0 - rank], world)

        class Args:
            pass
        ref = bench.run_reference(Args(), rank) if rank != 0 else "skipped"
        q.put((rank, got, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_replica():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict((r, (got, ref)) for r, got, ref in (q.get(timeout=10) for _ in range(world)))
    for r in range(world):
        assert res[r][0] == [2.0, 3.0, 10.0]  # element-wise max over both ranks
    assert res[1][1] is None  # the reference arm does no work off rank 0


def test_whole_job_rate_counts_every_replica():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(1e9, 1, 1.0) == pytest.approx(1e12)
    assert bench.whole_job_rate(1e9, 4, 2.0) == pytest.approx(2e12)
    assert bench.max_over_ranks([1, 2.5], 1) == [1.0, 2.5]


CHILD = r"""
import os, sys, torch, torch.distributed as dist
dist.init_process_group("gloo")
t = torch.tensor([float(os.environ["RANK"]) + 1.0])
dist.all_reduce(t)
assert os.environ["LOCAL_RANK"] == os.environ["RANK"]
assert os.environ["MASTER_ADDR"] == "127.0.0.1"
print("rank", os.environ["RANK"], "of", os.environ["WORLD_SIZE"], "sum", t.item(), flush=True)
dist.destroy_process_group()
"""


def test_bench_starts_its_own_ranks(capfd):
    """``bench.py --gpus N`` without torchrun starts N rank processes with the
    torchrun environment and a local rendezvous; here two gloo children
    rendezvous and all-reduce on the CPU."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    rc = bench.spawn_ranks(2, [sys.executable, "-c", CHILD])
    assert rc == 0
    out = capfd.readouterr().out
    assert "rank 0 of 2 sum 3.0" in out and "rank 1 of 2 sum 3.0" in out
