"""Host logic of bench.py's multi-replica mode, on CPU with gloo (world size 2)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, _ = bench._dist()
    secs = [0.5, 0.8][rank]
    out = (w, r, bench._max_over_ranks(secs, w), bench._job_throughput(100.0, secs, w))
    dist.barrier()
    dist.destroy_process_group()
    q.put(out)


def test_two_replicas_take_the_slowest_rank():
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
    for (w, r, mx, thr), rank in zip(res, (0, 1)):
        assert (w, r) == (2, rank)
        assert mx == pytest.approx(0.8)
        assert thr == pytest.approx(2 * 100.0 / 0.8)
