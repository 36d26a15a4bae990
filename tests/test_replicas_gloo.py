"""Multi-process path of the bench on CPU: two gloo ranks on 127.0.0.1.

The compress shards over independent (layer, batch, KV head) units with no
exchange, so N GPUs run N replicas.  What the ranks share is bookkeeping: each
takes its own layers, the job time is the slowest rank's, and the throughput
counts every rank's units.  These tests run that bookkeeping in two real
processes; no GPU is involved.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(elapsed[rank], world, "cpu")
        layers = bench.replica_layer_ids(rank, 4, 32)
        # every rank learns the others' layers to check they are disjoint
        gathered = [None] * world
        dist.all_gather_object(gathered, layers)
        dist.barrier()
        out[rank] = (ms, gathered)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_agree_on_the_slowest_time_and_split_the_layers():
    world = 2
    elapsed = [3.5, 7.25]   # rank 1 is the slow one
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, elapsed, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(90)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for r in range(world):
        ms, gathered = res[r]
        assert ms == max(elapsed)
        assert gathered[0] == [0, 1, 2, 3] and gathered[1] == [4, 5, 6, 7]
        assert not set(gathered[0]) & set(gathered[1])


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.replica_layer_ids(0, 4, 32) == [0, 1, 2, 3]


def test_job_throughput_counts_every_rank():
    # 2 ranks x 8 heads x 131072 keys per step, 10 steps in 5 ms
    v1 = bench.job_throughput(1, 8 * 131072, 10, 5.0)
    v2 = bench.job_throughput(2, 8 * 131072, 10, 5.0)
    assert v2 == 2 * v1
    assert v1 == pytest.approx(8 * 131072 * 10 / 5e-3)


def test_layers_wrap_when_ranks_outnumber_them():
    ids = [bench.replica_layer_ids(r, 4, 6) for r in range(2)]
    assert ids == [[0, 1, 2, 3], [4, 5, 0, 1]]
