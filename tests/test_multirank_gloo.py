"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

Sequences are independent, so ranks never exchange data; what they share is
the barrier and the max-over-ranks reduction of the timed region, and each
rank must draw a different batch of the same workload (weak scaling).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + rank, w)
    seed = bench.rank_seed(synth.WORKLOADS[4].seed, rank)
    inp = synth.generate([8], 1, 16, 16, seed=seed)
    out[rank] = (t, seed, float(inp.q.float().sum()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_and_seeds():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 11.0          # max over ranks
    assert out[0][1] != out[1][1]                  # distinct seeds
    assert out[0][2] != out[1][2]                  # distinct batches
