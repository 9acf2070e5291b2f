"""Multi-GPU is replicas only: every sequence's block, context KV and commit state are
independent, so N ranks run N independent copies and only the timing crosses ranks (a barrier
and a max of the elapsed time). This checks that host-side plumbing of bench.py with two
gloo ranks on the CPU."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(float(10 * (rank + 1)), w)   # rank 1 is the slowest
    out[rank] = m
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU path of the replica plumbing")
def test_two_gloo_ranks_agree_on_the_max_elapsed_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}
