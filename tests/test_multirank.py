"""The multi-GPU form of the benchmark is N replicas (the path shards by
tokens/rows with no exchange step): each rank runs the per-GPU workload on its
own seed, and rank 0 reports the bytes of all ranks over the slowest rank's
time.  The host-side bookkeeping is checked with two gloo ranks on CPU."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step, e2e = bench.reduce_max([1.0 + rank, 10.0 * (2 - rank)], world)
        w = synth.workloads(seed=rank)["gated_small"]
        q.put((rank, step, e2e, int(w.x(0, 1).astype(np.int64).sum())))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_own_seeds():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, step, e2e, _ in got:
        assert step == 2.0 and e2e == 20.0          # max over ranks, on every rank
    assert got[0][3] != got[1][3]                   # each rank draws its own inputs
    assert bench.aggregate_gbs(10**9, world, 2.0) == 1000.0


def test_single_rank_is_identity():
    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.aggregate_gbs(2 * 10**9, 1, 1.0) == 2000.0
