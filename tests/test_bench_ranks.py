"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank
draws its own batch, the job time is the slowest rank's, throughput counts
every rank's nodes, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    job_ms = bench.max_over_ranks(local_ms, "cpu")
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(2, rank))
    rc = bench.reference_arm(bench.parse_args(["--impl", "reference", "--steps", "1"]), world, rank) \
        if rank == 1 else 0
    out[rank] = (job_ms, seeds, rc)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        job_ms, seeds, rc = out[rank]
        assert job_ms == 20.0                    # the slowest rank sets the job time
        assert len(set(seeds)) == world          # every rank draws a different batch
        assert rc == 0                           # non-zero ranks leave the reference arm at once


def test_job_throughput_counts_all_ranks():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(512, 10, 4, 20.0) == pytest.approx(512 * 10 * 4 / 0.02)
    assert bench.max_over_ranks(3.0, "cpu") == 3.0
