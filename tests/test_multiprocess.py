"""The benchmark's multi-process plumbing on CPU (gloo, world size 2): the runs are
independent replicas with no data-path collective, so what crosses ranks is the barrier
around the timed region and the maximum of the ranks' times.  No GPU is involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(times[rank], w)
    bench.barrier(w)
    out[rank] = slowest
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_share_only_the_slowest_time(world):
    """Each rank sees the maximum of the ranks' times, which the benchmark divides the
    units of all ranks by (weak scaling: every rank runs its own full workload)."""
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    times = [1.25, 3.5]
    mp.start_processes(_worker, args=(world, _free_port(), times, out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 3.5, 1: 3.5}
    steps = 100
    value = steps * world / (max(times) / 1e3)
    assert value == pytest.approx(steps * world / 3.5e-3)


def _reference_worker(rank, world, port, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench

    class Args:
        steps, warmup, reference_seconds = 1, 0, 1.0
    if rank != 0:
        out[rank] = bench.run_reference(Args()) is None   # other ranks leave without work
    else:
        out[rank] = True


def test_reference_arm_runs_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_reference_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    assert dict(out) == {0: True, 1: True}
