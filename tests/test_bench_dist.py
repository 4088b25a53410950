"""The benchmark's multi-rank plumbing on CPU: world size 2 over gloo. Each rank is an
independent replica; the reported time is the maximum over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    assert bench.dist_env() == (world, rank, rank)
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    out[rank] = bench.reduce_max(1.5 + rank, world)
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max(3.25, 1) == 3.25


def test_reference_arm_nonzero_rank_does_no_work():
    import argparse

    import bench

    args = argparse.Namespace(steps=3, warmup=1)
    assert bench.run_reference(args, world=2, rank=1) is None


@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (4096, 14336, 4096)])
def test_algorithmic_bytes(M, N, K):
    import bench

    # 0.5 B per weight + 4 B of scale/min per 128 weights + x + y
    assert bench.w4a16_bytes(M, N, K) == N * K // 2 + N * K // 32 + 2 * M * K + 2 * M * N
    assert bench.weight_bytes(14336, 4096) == 31_195_136
