"""Host logic of bench.py for more than one rank, on CPU with gloo.

The codec has no cross-row exchange, so a multi-GPU run is independent
replicas: each rank times its own work between barriers and rank 0 reports the
maximum time (and the summed work). These tests run that aggregation with two
gloo ranks, and check that the reference arm does nothing off rank 0.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, ws = bench.init_dist("gloo")
    assert (r, ws) == (rank, world)
    bench.barrier()
    mx = bench.max_over_ranks(10.0 + 5.0 * rank)
    sm = bench.sum_over_ranks(1.0 + rank)
    # the reference arm runs on rank 0 only; other ranks return at once
    if rank != 0:
        class A:
            steps, warmup = 1, 3
        bench.run_reference(A())
    out[rank] = (mx, sm)
    torch.distributed.destroy_process_group()


def test_two_ranks_max_and_sum():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        assert out[0] == (15.0, 3.0) and out[1] == (15.0, 3.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5 and bench.sum_over_ranks(2.0) == 2.0
    assert bench.dist_env()[1] >= 1


def test_bytes_per_row_matches_layout():
    sys.path.insert(0, ROOT)
    import bench

    # D = 128, k8, v3, bf16: 512 B in + 128 + 48 codes + 8 + 8 + 8 scales
    assert bench.bytes_per_row(128, 8, 3, 2) == 712
    assert bench.bytes_per_row(512, 8, 5, 2) == 2976
