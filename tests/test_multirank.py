"""The N > 1 host logic of bench.py on two gloo ranks on the CPU: each rank
runs its own copy of the step (weak scaling, no data-path collective), the
reported time is the slowest rank's, the throughput counts every rank's work,
and only rank 0 runs the reference arm."""
import argparse
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)  # rank 1 is the slow one
        tflops = bench.whole_job_tflops(2e12, 3, world, slowest)
        ref = None
        if rank != 0:  # rank 0's reference arm would time the oracle; the others do no work
            ref = bench.run_reference(argparse.Namespace(steps=1, warmup=0), rank, world)
        out.put((rank, slowest, tflops, ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    results = {}
    try:
        for _ in range(2):
            rank, slowest, tflops, ref = q.get(timeout=180)
            results[rank] = (slowest, tflops, ref)
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.is_alive():
                pr.kill()
    assert [pr.exitcode for pr in procs] == [0, 0]
    for rank in (0, 1):
        slowest, tflops, _ = results[rank]
        assert slowest == 15.0
        # both ranks' work (2 x 3 steps x 2 TFLOP) over the slowest rank's 15 ms
        assert tflops == pytest.approx(2 * 3 * 2.0 / 15e-3)
    assert results[1][2] is None


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_tflops(1e12, 4, 1, 2.0) == pytest.approx(2000.0)
