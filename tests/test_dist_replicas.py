"""The N-GPU bench path is replicas only: each rank verifies its own
sequences, and the only cross-rank steps are the barrier and the max/sum of
the timings and token counts.  Those run here as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, _ = bench.dist_env()
    dist = bench.init_dist(ws, "gloo")
    bench.barrier(dist)
    elapsed = 1.5 + rank            # rank 1 is the slow one
    tokens = 10 * (rank + 1)
    t = bench.max_over_ranks(dist, elapsed)
    n = bench.sum_over_ranks(dist, tokens)
    out[rank] = (ws, r, t, n)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_tokens():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == (2, 0, 2.5, 30.0)
    assert out[1] == (2, 1, 2.5, 30.0)


def test_single_process_needs_no_process_group():
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    ws, rank, local = bench.dist_env()
    assert (ws, rank, local) == (1, 0, 0)
    assert bench.init_dist(ws, "gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0
