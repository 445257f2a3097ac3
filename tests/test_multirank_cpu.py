"""The benchmark's multi-rank logic on CPU (gloo, world size 2): replicas with
no data-path collective; the barrier and the max-over-ranks timing
reduction are the only collectives."""
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
    ws, r, local = bench.dist_setup(world)
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    elapsed = 10.0 + 5.0 * rank          # this rank's timed region (ms)
    mx = bench.reduce_max(elapsed, ws)
    # rank != 0 of the reference arm exits without work and prints nothing
    class A:
        warmup, steps, gpus = 3, 1, world
    if rank != 0:
        bench.run_reference(A, ws, rank)
    out[rank] = mx
    dist.destroy_process_group()


def test_two_rank_max_timing():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 15.0


def test_single_rank_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_setup(1)[0] == 1
    assert bench.reduce_max(3.5, 1) == 3.5
