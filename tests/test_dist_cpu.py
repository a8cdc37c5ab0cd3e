"""The bench's multi-rank host logic on CPU: two gloo ranks run bench.py's own process
group set-up, barrier and max-over-ranks reduction.

The path has no exchange step: under torchrun each rank runs an independent replica,
times its own steps, and the job's time is the slowest rank's.  These are the only
collectives involved, and what this test checks.
"""
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
    # CPU only wherever it runs: no GPU is visible to the ranks and the backend is gloo
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="", SL8_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup(None)
    assert dist.get_backend() == "gloo"
    assert (w, r, local) == (world, rank, rank)
    # a per-rank step time: the job's time is the slowest rank's
    got = bench.max_over_ranks(1.5 + 2.0 * rank, w)
    bench.barrier(w)
    out[rank] = got
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25, 1) == 2.25
    bench.barrier(1)
