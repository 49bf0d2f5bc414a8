"""The multi-GPU bench path on CPU: two gloo ranks run the host logic of bench.py's replica
mode (max over ranks, per-rank seeds, whole-job throughput) without a GPU."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.5, 2.25][rank]                       # rank 1 is the slow one
        got = bench.max_over_ranks(ms, world)
        q.put((rank, got, bench.replica_seed_base(rank), bench.job_throughput(64, world, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, s0, v0), (r1, ms1, s1, v1) = res
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 2.25                         # both ranks report the slowest
    assert s0 != s1                                   # replicas draw different inputs
    assert v0 == v1 == pytest.approx(64 * 2 / 2.25e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_throughput(64, 1, 1.0) == pytest.approx(64000.0)


def test_reference_arm_other_ranks_exit_without_output(capsys):
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), bench.WORKLOADS["small"], rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
