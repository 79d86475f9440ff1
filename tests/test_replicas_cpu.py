"""The N > 1 path of the bench, on CPU with gloo (world size 2): every rank
runs its own replica (the path shards by token with no exchange step), the
timings are reduced with a max over ranks, and throughput is whole-job."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + rank, 30.0 - rank, 1.0 * (rank + 1)]
        got = bench.max_over_ranks(local, world, device="cpu")
        q.put((rank, got, bench.whole_job_throughput(256, 100, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
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
    for rank, got, thr in out:
        assert got == [11.0, 30.0, 2.0]
        assert thr == pytest.approx(256 * 100 * 2 / 11e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.0, 2.0], 1) == [1.0, 2.0]
