"""The benchmark's process handling on CPU.

The decode runs on one GPU only (its conv kernels share weight tiles inside a
CTA cluster with multicast TMA loads, issued only in one-GPU processes), so a
multi-GPU launch of the decode stops before any CUDA call; the reference arm
(the CPU oracle) runs on rank 0 alone when launched under torchrun, which is
checked here with two gloo ranks on 127.0.0.1.
"""

import os
import socket
import sys

import pytest
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
        # the decode arm refuses a multi-process launch on every rank
        try:
            bench.check_one_gpu(world, world)
            out[f"refused{rank}"] = False
        except SystemExit as e:
            out[f"refused{rank}"] = "one GPU" in str(e)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_both_refuse_the_decode():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out["refused0"] is True and out["refused1"] is True


def test_one_gpu_check():
    import bench
    bench.check_one_gpu(1, 1)
    for gpus, world in ((2, 1), (1, 2), (8, 8)):
        with pytest.raises(SystemExit):
            bench.check_one_gpu(gpus, world)


def test_bench_main_refuses_before_cuda(monkeypatch):
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2"])
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "one GPU" in str(e.value)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 3
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
