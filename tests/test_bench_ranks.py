"""The multi-rank side of bench.py on the CPU: two gloo ranks.

On N GPUs every rank runs an independent replica ("replicas only": the
attention path needs no exchange between GPUs).  What the ranks share is
the reporting:
- the slowest rank's time, reduced with MAX over the ranks;
- the whole-job throughput, which counts every replica's work;
- rank 0 alone prints, and the reference arm runs on rank 0 only."""
import io
import os
import socket
import contextlib

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        buf = io.StringIO()
        args = type("A", (), {"steps": 1, "warmup": 0, "ref_rows": 4})()
        if r != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(args, w, r, local)   # rank != 0: no work, no output
        out[rank] = (w, r, local, ms, buf.getvalue())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for rank in range(world):
        w, r, local, ms, printed = out[rank]
        assert (w, r, local) == (world, rank, rank)
        assert ms == 15.0            # every rank sees the slowest rank's time
    assert out[1][4] == ""           # the reference arm stays silent on rank 1


def test_job_throughput_counts_every_replica():
    one = bench.job_throughput(1, 1.0e12, 10, 100.0)
    two = bench.job_throughput(2, 1.0e12, 10, 100.0)
    assert one == pytest.approx(100.0) and two == pytest.approx(2 * one)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
