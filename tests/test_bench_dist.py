"""Host-side logic of the N > 1 benchmark path (replicas): the barrier, the max
over ranks and the whole-job value, on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    bench.barrier(world)
    local_seconds = 1.0 + rank            # rank 1 is the slow one
    t = bench.reduce_max(local_seconds, world)
    v = bench.aggregate_value(flops_per_step=1e12, steps=10, world=world, max_seconds=t)
    out[rank] = (t, v, bench.dist_env())
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        t, v, env = out[rank]
        assert t == 2.0                       # the slowest rank's time
        assert v == pytest.approx(world * 10 * 1e12 / 2.0 / 1e12)
        assert env == (world, rank, rank)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate_value(2e12, 5, 1, 2.0) == pytest.approx(5.0)


def test_warmup_and_gpus_arguments_are_checked():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2"])        # WORLD_SIZE is 1 here
