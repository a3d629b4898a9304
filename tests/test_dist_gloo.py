"""The multi-rank logic of bench.py on CPU: two gloo ranks, barrier,
max-over-ranks timing and the weak-scaling whole-job value."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # rank-dependent "times": the slowest rank sets the job time
    t = 1.0 + rank
    t_max = bench.max_over_ranks(t, w)
    value = bench.weak_scaling_value(10.0, w, t_max)
    out[rank] = (t_max, value)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: (2.0, 10.0), 1: (2.0, 10.0)}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(10.0, 1, 2.0) == 5.0
