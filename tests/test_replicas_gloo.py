"""The multi-GPU path of bench.py is N independent replicas (the method has no exchange
step).  Its host-side logic runs here as two gloo ranks on the CPU: each rank draws
its own seeded layers, the slowest rank's time is the job's time, and the job's
ms per layer divides it by every layer all ranks processed."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank            # rank 1 is the slow one
        job = bench.reduce_max(local_ms, dist)
        out.put((rank, bench.replica_layers(rank, 2), job, bench.job_ms_per_layer(job, 10, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    layers = [r[1] for r in res]
    assert layers == [[0, 1], [2, 3]]                 # disjoint seeded layers per rank
    assert all(r[2] == 150.0 for r in res)            # every rank sees the slowest rank's time
    assert all(r[3] == pytest.approx(150.0 / 20) for r in res)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.replica_layers(0, 3) == [0, 1, 2]
    assert bench.job_ms_per_layer(30.0, 10, 1) == 3.0
