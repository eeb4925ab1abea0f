"""The N>1 bench path on CPU: two gloo ranks, each an independent replica of
the decode step (no data-path collective), joined only by the barrier and the
max-over-ranks timing reduction bench.py uses.  Also checks that replicas draw
different step inputs (seed offset by rank) while sharing the workload shape."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads as W
    r, w, local, pg = bench.dist_setup(None)
    assert (r, w) == (rank, world) and pg is not None
    bench.barrier(pg)
    t = bench.max_over_ranks(pg, 1.0 + rank)            # each rank's own step time
    wl = W.TINY
    q, k, v = W.device_q(wl, "cpu", salt=rank)          # replica inputs differ by rank
    out[rank] = (t, float(q.float().sum()), tuple(wl.seq_lens()))
    pg.destroy_process_group()


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.0                # max over ranks
    assert out[0][1] != out[1][1]                       # independent replicas
    assert out[0][2] == out[1][2]                       # same workload shape
