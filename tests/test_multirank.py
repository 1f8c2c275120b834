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


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    """The reference arm's one JSON line: the oracle timed on the host cores, with the keys the
    bench contract names."""
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class Args:
        workload, cache, steps, warmup, ref_seconds = "tiny", "bf16", 2, 3, 0.25

    bench.run_reference(Args())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "tiny"


def test_reference_sample_fits_its_budget():
    """Each step's sample fits the per-step budget at the measured rate (at least one row), so
    that a run of any step count stays within a few minutes."""
    from workloads import make_case
    for name in ("tiny", "batch", "ragged"):
        case = make_case(name)
        lens = case.seq_lens.numpy()
        rate = 0.4e9
        for seconds in (0.01, 0.1, 1.0):
            rows, _, threads = bench._reference_sample(case, seconds, rate)
            assert 1 <= len(rows) <= case.B * case.Hq and 1 <= threads <= len(rows)
            cost = [lens[b] * case.D * 4.0 / rate for b, _ in rows]
            per_thread = max(sum(cost[i::threads]) for i in range(threads))
            assert len(rows) == 1 or per_thread <= seconds + 1e-12
