"""The N > 1 benchmark path on CPU: two gloo ranks, each an independent replica.

Checks the whole-job aggregation (max time over ranks, summed work) and that
each rank's batch is its own seeded workload whose tables the host allocator
builds independently (sequence sharding, no data-path collective).
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as wl
        from paged_kv_cache_88_gb300 import binding as bd
        ms = 10.0 + 5.0 * rank
        res = bench.aggregate_ranks(ms, 100.0 * (rank + 1), 32.0, "cpu")
        w = wl.make_workload(2, num_layers=1, seed=bench.rank_seed(2, rank))
        pool = bd.Pool(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, initial_free_order=w.free_order)
        first = pool.alloc(3)
        q.put((rank, res, int(w.context_lens.sum()), first))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, (ms, kv, seqsteps), tokens, first in out:
        assert ms == 15.0                      # slowest rank's time
        assert kv == 300.0                     # work summed over ranks
        assert seqsteps == 64.0
    # different ranks serve different batches (weak scaling)
    assert out[0][2] != out[1][2] and out[0][3] != out[1][3]


def test_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(3.0, 7.0, 9.0) == (3.0, 7.0, 9.0)
