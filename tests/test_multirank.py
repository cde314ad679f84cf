"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

Each rank decodes its own clip (no exchange on the data path); the step time
is the slowest rank's and the value is the whole job's frames/s.  The
reference arm runs on rank 0 only.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(100.0 + 50.0 * rank, dist, "cpu")
        value = bench.weak_scaling_value(ms, world, 121)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_weak_scaling():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 150.0
        assert value == pytest.approx(2 * 121 / 0.150)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.weak_scaling_value(1000.0, 1, 121) == pytest.approx(121.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 3
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
