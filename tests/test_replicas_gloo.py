"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank is an
independent replica; only the job aggregate (token sum, slowest rank's time) crosses
ranks, and rank 0 alone reports."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    tokens, seconds = bench.reduce_job(dist, tokens=100.0 + rank, seconds=1.0 + 0.5 * rank)
    bench.barrier(dist)
    results[rank] = (tokens, seconds)
    dist.destroy_process_group()


def test_reduce_job_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        assert results[r] == pytest.approx((201.0, 1.5))


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_job(None, 7.0, 2.0) == (7.0, 2.0)
