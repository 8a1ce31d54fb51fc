"""The bench's multi-rank combination (max time, summed bytes) on two gloo
ranks on the CPU: each rank runs an independent batch, no data-path
collective; only the final timing reduction crosses ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, nbytes = bench.reduce_over_ranks(10.0 + rank, 1000 * (rank + 1), torch.device("cpu"))
    q.put((rank, ms, nbytes))
    dist.destroy_process_group()


def test_reduce_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, nbytes in got:
        assert ms == 11.0 and nbytes == 3000.0


def test_single_process_is_identity():
    import bench
    assert bench.reduce_over_ranks(5.0, 7) == (5.0, 7.0)
