"""The benchmark's multi-rank host logic on CPU: two gloo ranks, as torchrun
would start them for `bench.py --gpus 2` (replicas, barrier, max over ranks),
and the reference arm's rank rule (rank 0 works, the others return nothing)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import argparse
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = [2.5, 7.0][rank]
        bench.barrier(world)
        out[rank] = bench.barrier_max(x, world)
        args = argparse.Namespace(workload="llama32k", steps=1, warmup=0)
        if rank != 0:  # non-zero ranks of the reference arm exit without work
            assert bench.reference_arm(args, rank, world) is None
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 7.0, 1: 7.0}


def test_single_rank_is_identity():
    import bench
    assert bench.barrier_max(3.25, 1) == 3.25
    bench.barrier(1)
