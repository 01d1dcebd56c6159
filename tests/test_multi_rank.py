"""The N > 1 host path of bench.py on CPU: world size 2 over gloo (127.0.0.1).

Each rank runs an independent replica (the path shards by request and KV head with no
exchange); the only cross-rank operations are the barrier around the timed region and
the max over ranks of the elapsed time, which these tests exercise."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
        q.put((rank, r, w, t))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_on_gloo():
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
    assert [(r, w) for _, r, w, _ in res] == [(0, 2), (1, 2)]
    assert all(t == 15.0 for *_, t in res)        # every rank sees the slowest rank's time


def _ref_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from kvd_inputs import get

    class A:
        steps, warmup, cpu_budget = 1, 3, 0.05

    line = bench.reference_arm(A, get("tiny"), rank, world)
    q.put((rank, None if line is None else line["impl"]))


def test_reference_arm_prints_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    assert sorted(q.get(timeout=10) for _ in range(2)) == [(0, "reference"), (1, None)]
