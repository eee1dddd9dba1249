"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

The convolution path needs no exchange between GPUs (each rank runs an
independent replica), so the only multi-rank logic is the benchmark's
aggregation: the step time is the maximum over ranks, and only rank 0 prints.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_time = 10.0 + 5.0 * rank        # rank 1 is the slow one
    got = bench.reduce_max(local_time, world)
    r, w, _ = bench.dist_env()
    q.put((rank, got, r, w))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [(r[2], r[3]) for r in res] == [(0, 2), (1, 2)]


def _ref_worker(rank, world, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    class A:
        steps, warmup, gpus = 1, 3, world
    q.put((rank, bench.bench_reference(A()) if rank != 0 else "rank0"))


def test_reference_arm_non_zero_ranks_exit_without_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_ref_worker, args=(1, 2, q))
    p.start()
    p.join(timeout=60)
    assert p.exitcode == 0
    assert q.get(timeout=10) == (1, 0)
