"""The benchmark's multi-rank path on CPU (gloo, world size 2): every rank runs its own
replica, the step time is the slowest rank's, and the job's throughput counts every
rank's bytes.  No GPU and no collective on the data path."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.5, 7.25][rank]
        out[rank] = bench.max_over_ranks(local_ms, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        assert dict(out) == {0: 7.25, 1: 7.25}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.0, None, "cpu") == 4.0


def test_weak_scaling_counts_every_rank():
    one = bench.weak_scaling_gbs(92_097_048, 1, 0.0282)
    assert one == pytest.approx(92_097_048 / 28.2e-6 / 1e9)
    assert bench.weak_scaling_gbs(92_097_048, 4, 0.0282) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, steps, warmup, ref_seconds = "tiny", 1, 3, 0.25

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
