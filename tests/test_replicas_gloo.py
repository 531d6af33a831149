"""Multi-replica host logic of bench.py on CPU with the gloo backend
(world size 2): each rank decodes its own batch (weak scaling, no collective
on the data path); the job's time is the slowest rank's and its work the sum
over ranks."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from paged_kv_cache_124_gb300 import inputs as I
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    # each replica draws its own batch
    seed = bench.replica_seed(0, r)
    sc = I.batch64_8b(seed)
    first_alloc = [op for op in sc.ops if op[0] == "alloc"][:4]
    elapsed = 1.0 + r            # rank 1 is slower
    units = 100 * (r + 1)
    t, u = bench.reduce_timing(elapsed, units, w)
    bench.barrier(w)
    results[rank] = (seed, first_alloc, t, u)
    dist.destroy_process_group()


def test_two_gloo_replicas_reduce_time_and_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    (s0, a0, t0, u0), (s1, a1, t1, u1) = results[0], results[1]
    assert s0 != s1 and a0 != a1                 # different batches per replica
    assert t0 == t1 == 2.0                       # slowest rank
    assert u0 == u1 == 300.0                     # total work


def test_single_process_needs_no_process_group():
    import bench
    assert bench.reduce_timing(3.5, 7, 1) == (3.5, 7.0)
    assert not torch.distributed.is_initialized()
