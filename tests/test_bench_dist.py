"""Host logic of the multi-rank benchmark (replicas, weak scaling), run as
two gloo ranks on the CPU: the timed region is the max over ranks, the value
counts every rank's bytes, and the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.5, 7.25][rank]
        got = bench.max_over_ranks(mine, dist, "cpu")
        results[rank] = got
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), results), nprocs=2, join=True,
                           start_method="spawn")
        assert dict(results) == {0: 7.25, 1: 7.25}


def test_job_value_counts_every_rank():
    # 2 ranks x 10 steps x 1 GB in 5 ms (the slower rank) -> 4000 GB/s
    assert bench.job_gbs(2, 10**9, 10, 5.0) == pytest.approx(4000.0)
    assert bench.job_gbs(1, 10**9, 10, 5.0) == pytest.approx(2000.0)
    assert bench.max_over_ranks(1.5) == 1.5


def test_reference_arm_only_on_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
