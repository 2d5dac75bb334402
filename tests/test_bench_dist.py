"""The benchmark's multi-rank bookkeeping on CPU: world_size 2 over gloo.

Each rank runs its own replica of the workload; the only cross-rank traffic
is a barrier and a max-reduction of the timed region (host scalars), and the
reported throughput counts the work of all ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier()
    t = bench.max_over_ranks(1.0 + rank)  # rank 1 is the slow one
    out[rank] = t
    bench.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 2.0


def test_single_rank_is_identity():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_env()[0] == 1
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5) == 3.5


def test_rotation_count_covers_twice_l2():
    import bench
    l2 = 126 * 2 ** 20
    for per_set in (1 << 20, 64 << 20, 200 << 20, 400 << 20):
        n = bench.rotation_count(per_set, l2, cap=64)
        assert n >= 2
        if per_set * 64 > 2 * l2:
            assert n * per_set > 2 * l2
