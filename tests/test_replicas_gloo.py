"""The multi-GPU path is independent replicas (the forward pass has no
exchange step).  This checks its host logic with two gloo ranks on CPU: the
barrier, the max-over-ranks of the timed interval and the whole-job token
count `bench.py` reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        bench.barrier(w)
        elapsed = 1.0 + rank           # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, w)
        tokens_per_rank = 48 * 10
        value = tokens_per_rank * w / slowest
        q.put((r, lr, w, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, lrank, world, slowest, value) in enumerate(res):
        assert (rank, lrank, world) == (r, r, 2)
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(48 * 10 * 2 / 2.0)
