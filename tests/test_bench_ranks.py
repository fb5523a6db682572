"""The bench's multi-rank plumbing on CPU (gloo, world size 2): the layer runs as
independent replicas, one per GPU, so the only cross-rank step is taking the slowest
rank's step time; the whole-job value then counts every rank's work.  No GPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        mine = 0.150 + 0.010 * rank  # ms per step on this rank
        worst = bench.combine_ranks(mine, world, torch.device("cpu"))
        out[rank] = (worst, bench.job_value(worst, world, 4.64e9))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        worst, value = out[r]
        assert worst == pytest.approx(0.160)
        assert value == pytest.approx(world * 3 * 4.64e9 / (0.160e-3) / 1e9)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(0.2, 1, None) == 0.2
    assert bench.job_value(0.2, 1, 1e9) == pytest.approx(3 * 1e9 / 0.2e-3 / 1e9)
