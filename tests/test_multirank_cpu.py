"""The N > 1 path of bench.py on CPU: two gloo ranks, replica seeding, barrier and the
max-over-ranks timing.  The path shards by sequence with no exchange (replicas only), so the
only cross-rank operations are the barrier and the max reduction of the step time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import argparse

    import torch.distributed as dist

    import bench
    args = argparse.Namespace(impl="reference")
    w, r, _ = bench.dist_setup(args)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports a different step time; every rank must see the max
    m = bench.dist_max(1.5 + rank, w, "cpu")
    out[rank] = m
    # replicas draw different batches (seed offset by rank), same shapes
    import workloads
    q, kv, kw = workloads.config_lengths(2, 1002 + 7919 * rank)
    out[world + rank] = float(sum(kv))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Array("d", 2 * world)
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert list(out[:world]) == [2.5, 2.5]
    assert out[world] != out[world + 1]
