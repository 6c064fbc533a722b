"""The bench's multi-rank bookkeeping on CPU: two gloo ranks on 127.0.0.1.

The decode path has no data-path collective (replicas only); what runs on
several ranks is the timing aggregation: the job time is the slowest rank's,
and throughput counts every replica's tokens."""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]           # rank 1 is the slower replica
        m = bench.max_over_ranks(ms, world, "cpu")
        out.put((rank, m, bench.replica_throughput(1000, m, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # 2 replicas x 1000 tokens in 5 ms
    assert all(r[2] == pytest.approx(2 * 1000 / 5e-3) for r in res)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.replica_throughput(100, 2.0, 1) == pytest.approx(5e4)
