"""The N > 1 host path (independent replicas, max-over-ranks timing) with two
gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_attention_decode_step_gb300 import inputs, replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "timed" a different duration; the job time is the max
        local = [1.0 + rank, 10.0 - rank]
        dist.barrier()
        got = replicas.max_over_ranks(local, dist)
        seeds = [replicas.rank_layer_seed(inputs.SEED_DECODE_STACK, l, rank) for l in range(34)]
        allseeds = [None] * world
        dist.all_gather_object(allseeds, seeds)
        out[rank] = (got, allseeds)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_distinct_seeds():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        got, allseeds = out[r]
        assert got == [2.0, 10.0]
        flat = [s for rs in allseeds for s in rs]
        assert len(set(flat)) == len(flat)  # no two ranks share a layer's inputs


def test_single_process_passthrough_and_aggregate():
    assert replicas.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert replicas.rank_layer_seed(inputs.SEED_DECODE_STACK, 5, 0) == 3005
    # weak scaling: 2 ranks x 1 GB in 0.5 s (slowest rank) -> 4 GB/s
    assert replicas.job_throughput(1e9, 2, 0.5) == 4e9
