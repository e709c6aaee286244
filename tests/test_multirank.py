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


# ---- split-KV of one long sequence across ranks (host logic) ----------------


def _split_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np
        from oracle import mla as O
        from mla_latent_kv_74_b300 import multigpu
        rng = np.random.default_rng(7)  # the same inputs on every rank
        H, d_h, d_c, d_r, bs, Hq = 3, 4, 8, 2, 4, 2
        nb = 40
        cache = rng.standard_normal((nb, bs, d_c + d_r))
        bt = rng.permutation(nb)[:2 * 16].reshape(2, 16)
        sl = np.array([61, 23])
        qn = rng.standard_normal((2, Hq, H, d_h))
        qr = rng.standard_normal((2, Hq, H, d_r))
        W1 = rng.standard_normal((H, d_h, d_c))
        W2 = rng.standard_normal((H, d_h, d_c))
        first, end = multigpu.block_range(rank, world, bt.shape[1])
        # the oracle stands in for this rank's mla_decode_blocks call
        _, o, lse = O.mla_decode_blocks(qn, qr, cache, bt, sl, W1, W2, Hq, first, end)
        o_all, lse_all = multigpu.gather_pieces(torch.tensor(o), torch.tensor(lse), dst=0)
        if rank == 0:
            o_m, lse_m = O.combine_pieces(o_all.numpy(), lse_all.numpy())
            _, o_ref, lse_ref = O.mla_decode(qn, qr, cache, bt, sl, W1, W2, Hq)
            q.put((rank, float(np.abs(o_m - o_ref).max()),
                   float(np.abs(lse_m - lse_ref).max()), (first, end)))
        else:
            q.put((rank, o_all is None and lse_all is None, None, (first, end)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_block_ranges_gathered_and_merged_equal_the_whole_decode(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = {r: rest for r, *rest in (q.get(timeout=10) for _ in range(world))}
    assert res[0][0] < 1e-12 and res[0][1] < 1e-12  # merged pieces == whole decode
    for r in range(1, world):
        assert res[r][0] is True  # only the destination rank receives the pieces
    ranges = [res[r][2] for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == 16
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))


def test_block_range_partitions_the_blocks():
    import sys
    sys.path.insert(0, ROOT)
    from mla_latent_kv_74_b300 import multigpu
    for n in (0, 1, 5, 16, 2049):
        for world in (1, 2, 3, 8):
            rs = [multigpu.block_range(r, world, n) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            assert max(e - f for f, e in rs) - min(e - f for f, e in rs) <= (n + world - 1) // world
    with pytest.raises(ValueError):
        multigpu.block_range(2, 2, 10)
