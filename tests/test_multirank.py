"""The N>1 bench path on CPU: two gloo ranks, replicas with their own seeds,
job time = max over ranks (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from sparse_paged_kv_locks_gb300 import workload as W
    bench.dist_init(world, "gloo")
    r, w, lr = bench.dist_env()
    spec = bench.rank_spec(W.SPECS["tiny_4k"], r)
    t = bench.reduce_max(1.0 + r)          # rank 1 is the slow one
    bench.barrier()
    out[rank] = (r, w, spec.seed, t)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][:2] == (0, 2) and out[1][:2] == (1, 2)
    assert out[0][2] != out[1][2]                  # independent replicas
    assert out[0][3] == out[1][3] == 2.0           # max over ranks
