"""Multi-rank host logic of bench.py on CPU: world size 2 over gloo.

The verify step shards by request with no collective on the data path
(replicas); the only cross-rank operations are the barrier around the timed
region and the max over ranks of the step time, checked here.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w)          # rank 1 is the slow one
    bench.barrier(w)
    q.put((rank, t))
    dist.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import bench

    class A:
        workload = "tiny"
        warmup = 3
        steps = 3
        gpus = 2
    bench.run_reference(A, rank=1, world=2, local=1)
    assert capsys.readouterr().out == ""
