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
    """Each step's sample fits the per-step budget at the measured rate, or, where the first row
    alone outlasts it, the time of that row (the other threads take rows beside it), so that a
    run of any step count stays within a few minutes."""
    from workloads import make_case
    for name in ("tiny", "batch", "ragged"):
        case = make_case(name)
        lens = case.seq_lens.numpy()
        rate = 0.4e9
        for seconds in (0.001, 0.01, 0.1, 1.0):
            rows, _, threads = bench._reference_sample(case, seconds, rate)
            assert 1 <= len(rows) <= case.B * case.Hq and 1 <= threads <= len(rows)
            cost = [lens[b] * case.D * 4.0 / rate for b, _ in rows]
            per_thread = max(sum(cost[i::threads]) for i in range(threads))
            assert per_thread <= max(seconds, cost[0]) + 1e-12


def test_reference_sample_keeps_every_thread_busy_on_long_rows(monkeypatch):
    """One row of the long-context workload outlasts a short per-step budget: the step still
    takes one row per host thread (the same wall time as one row), not a single row."""
    import types
    import torch
    monkeypatch.setattr(bench.os, "cpu_count", lambda: 16)
    # the long-context shape (only the lengths and sizes matter to the sample)
    case = types.SimpleNamespace(B=4, Hq=64, D=128, seq_lens=torch.full((4,), 131072, dtype=torch.int32))
    rate = 0.4e9
    one_row = 131072 * case.D * 4.0 / rate
    rows, _, threads = bench._reference_sample(case, one_row / 2, rate)
    assert len(rows) == 16 and threads == 16


def test_roofline_picks_the_binding_roof():
    """A tensor-core call reports the roof that takes longer at its peak: HBM for a long table
    with few rows per group, the tensor cores for a short table with many."""
    from workloads import algorithmic_bytes, make_prefill_case
    peaks = {"hbm_gbs": 6789.6, "bf16_tflops": 1874.7, "source": "measured"}

    class Args:
        workload, cache = "long", "bf16"

    spec = dict(B=1, Hq=8, Hkv=1, D=128, P=16, lens=("fixed", 1), seed=0)
    for L, q_len, want in ((65536, 8, "hbm"), (2048, 1024, "tensor")):
        case = make_prefill_case(spec, [q_len], [L])
        ms = 1.0
        gbs = algorithmic_bytes(case)["total"] / (ms * 1e-3) / 1e9
        r = bench._roofline(Args, case, q_len, False, 128, peaks, gbs, ms)
        assert r["bound"] == want and r["secondary"]["bound"] != want
        t_hbm = algorithmic_bytes(case)["total"] / (peaks["hbm_gbs"] * 1e9)
        t_tensor = bench.causal_flops(case) / (peaks["bf16_tflops"] * 1e12)
        assert (t_hbm > t_tensor) == (want == "hbm")
        frac = {r["bound"]: r["frac"], r["secondary"]["bound"]: r["secondary"]["frac"]}
        assert abs(frac["hbm"] - t_hbm / (ms * 1e-3)) < 1e-3 and abs(frac["tensor"] - t_tensor / (ms * 1e-3)) < 1e-3
