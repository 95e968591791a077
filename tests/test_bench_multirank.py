"""The benchmark's multi-rank bookkeeping with two gloo ranks on the CPU: timings reduce to
the slowest rank, and replicas add their work."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 5.0 - rank, 7.0]
    out[rank] = bench.max_over_ranks(local, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 5.0, 7.0]


def test_replica_throughput_counts_every_rank():
    # 4 replicas, 10 steps of 1e12 FLOP each, slowest rank 2 s -> 2e13 FLOP/s
    assert bench.replica_throughput(4, 10, 1e12, 2.0) == 2e13
    assert bench.replica_throughput(1, 10, 1e12, 2.0) == 5e12
