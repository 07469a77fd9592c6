"""CPU test of the N > 1 path of bench.py with two gloo ranks.

The product needs no exchange between GPUs, so N GPUs run N independent
replicas; the only cross-rank logic is the barrier, the max over ranks of the
timed region and the sum of the work all ranks did. This runs that logic on
two host processes (gloo backend, 127.0.0.1)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        elapsed, flops = bench.reduce_over_ranks(1.5 + rank, 1e12 * (rank + 1), torch.device("cpu"))
        w, r, l = bench.dist_env()
        args = bench.main.__globals__["argparse"].Namespace(
            only=None, steps=3, warmup=3, reference_budget=1.0)
        ref = bench.run_reference(args) if rank == 1 else "skipped"
        out[rank] = (elapsed, flops, w, r, l, ref)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        elapsed, flops, w, r, l, ref = out[rank]
        assert elapsed == 2.5, "timed region is the slowest rank's"
        assert flops == 3e12, "work is summed over ranks"
        assert (w, r, l) == (world, rank, rank)
    assert out[1][5] is None, "only rank 0 runs the reference arm"
