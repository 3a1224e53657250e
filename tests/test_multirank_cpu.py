"""The N > 1 control path of bench.py on CPU: two gloo ranks (127.0.0.1)
agree on the slowest rank's time and on the whole-job throughput, and the
reference arm does its work on rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_setup()
        my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        dist.barrier()
        worst = bench.max_over_ranks(my_ms, dist, torch.device("cpu"))
        value = bench.whole_job_tflops(w, 10**12, 4, worst)
        results[rank] = (w, r, l, worst, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_use_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for rank in range(2):
        w, r, l, worst, value = results[rank]
        assert (w, r, l) == (2, rank, rank)
        assert worst == 15.0
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert abs(value - 2 * 4 * 1.0 / 15e-3) < 1e-9


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert abs(bench.whole_job_tflops(1, 2 * 10**12, 10, 1000.0) - 20.0) < 1e-12


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 3, "warmup": 3})()
    rank, res = bench.run_reference(args, bench.by_name("tiny_mha_d64"))
    assert rank == 1 and res is None
