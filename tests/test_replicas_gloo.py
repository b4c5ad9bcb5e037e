"""Host logic of the N > 1 benchmark path on CPU: two gloo ranks, each an
independent replica, combine their timings as max over ranks and their work
as a sum (weak scaling; no collective on the data path)."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 1.0 + rank          # rank 1 is the slower replica
        units = 100.0 * (rank + 1)
        bench.barrier()
        q.put((rank, bench.reduce_max_sum(elapsed, units)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_sum_of_work():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    for r in (0, 1):
        assert got[r] == (2.0, 300.0)


def test_single_process_is_identity():
    import bench

    assert bench.reduce_max_sum(1.5, 7.0) == (1.5, 7.0)
