"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks (replicas, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, "cpu", world)
        dist.barrier()
        out[rank] = (slowest, bench.job_tflops(world, 4, 1e12, slowest))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        slowest, tflops = out[r]
        assert slowest == 15.0
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert tflops == pytest.approx(2 * 4 * 1.0 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, "cpu", 1) == 3.5
    assert bench.job_tflops(1, 10, 2e12, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1))

    class Args:
        steps, warmup, workload, density, heads = 2, 1, "tiny", None, None
    assert bench.reference_arm(Args()) == 0
    assert not called
