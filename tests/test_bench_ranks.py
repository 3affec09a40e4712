"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the
barrier, the max over ranks of the step time, the whole-job throughput of
replicas, and the reference arm doing no work on ranks other than 0."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, max_over_ranks = bench.rank_sync(world, torch.device("cpu"))
        times = [3.5, 7.25]
        barrier()
        out[rank] = max_over_ranks(times[rank])
        barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert dict(out) == {0: 7.25, 1: 7.25}


def test_single_rank_sync_is_identity():
    import bench
    barrier, max_over_ranks = bench.rank_sync(1, torch.device("cpu"))
    barrier()
    assert max_over_ranks(1.5) == 1.5


def test_job_throughput_counts_every_replica():
    import bench
    # 8.64 TFLOP per rank and step, 8.7 ms per step on the slowest rank
    assert bench.job_tflops(8.64e12, 1, 8.7) == pytest.approx(993.1, rel=1e-4)
    assert bench.job_tflops(8.64e12, 4, 8.7) == pytest.approx(4 * 993.1, rel=1e-4)


def test_reference_arm_idles_on_other_ranks(monkeypatch):
    import bench
    import usp_workloads as W
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 0

    def no_oracle(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")

    monkeypatch.setattr(bench, "oracle_sample", no_oracle)
    assert bench.run_reference(Args(), W.TINY) == 0
