"""Host logic of the multi-GPU bench path (independent replicas), on CPU with
gloo, world size 2: the timed region is the max over ranks, the value counts
every rank's tokens, and only rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + rank * 5.0)
        v = bench.throughput(4096, 10, world, t)
        class A:
            steps, warmup, ref_budget, ref_tokens = 1, 0, 0.2, 1
        r = bench.bench_reference(A, None) if rank != 0 else 0
        out[rank] = (t, v, r)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_host_logic():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0                # max over ranks
    assert abs(out[0][1] - 4096 * 10 * 2 / 0.015) < 1e-6  # whole-job tokens/s
    assert out[1][2] == 0                                 # non-zero ranks skip the reference arm


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.throughput(100, 4, 1, 2.0) == pytest.approx(200000.0)
