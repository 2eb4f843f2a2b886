"""The N>1 path of bench.py on CPU: two gloo ranks, each an independent replica (the
attention path has no exchange step).  The whole-job number takes the max step time
over ranks and the work of all ranks; the reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.reduce_step_time(10.0 + 5.0 * rank, world)
    out[rank] = (ms, bench.job_throughput(1e12, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_sums_work():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, tflops = out[rank]
        assert ms == pytest.approx(15.0)                  # slowest rank
        assert tflops == pytest.approx(2 * 1e12 / 15e-3 / 1e12)  # both ranks' work


class _Args:
    gpus, steps, warmup, causal, N, B, H, d, which = 2, 1, 0, False, 256, None, 1, 64, "step"


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(_Args())
    assert capsys.readouterr().out == ""
