"""Benchmark: paged GQA decode attention on GB300 through the C-ABI library.

One step = one call of the whole hot path (plan, page-table walk, TMA page
gather, scores, online softmax, PV, split epilogue, merge) over one batch of
seeded synthetic inputs resident in HBM.  L2 is flushed before every timed step,
outside the step's event pair: a 2 x L2-size buffer is rewritten, then a second
2 x L2-size buffer is read, so that the step starts with a cold L2 holding clean
lines only (the flush's own dirty lines are written back before the step, not
inside it).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--cache bf16|fp8]
                    [--impl pkv|reference]

The default workload is the long-context one (B=4, Hq=64, Hkv=8, D=128, 16-key pages,
131072 keys per sequence, ~2.1 GB of K/V): the largest single-GPU configuration, the one
whose split count and merge matter most.  After the headline, every decode workload is
timed once more on both caches in the same process (`per_config`).

Prints one JSON line (rank 0).  `value` is achieved GB/s of algorithmic bytes
(K and V of the valid keys, q, out, lse, used block-table entries, lengths)
summed over all ranks, divided by the max over ranks of the time per step.
`--cache fp8` runs the same workload over an fp8 (e4m3) cache with per-(token, kv
head) power-of-two scales, quantised on the device before timing; its algorithmic
bytes count one byte per K/V element plus the scales.
`--impl reference` times the CPU fp64 oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attn: µs/call, achieved HBM GB/s and % of GB300 peak"
NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = ["paged_kv_gqa_gb300/csrc/decode_kernel.cuh", "paged_kv_gqa_gb300/csrc/ptx.cuh",
                  "paged_kv_gqa_gb300/csrc/plan.h", "paged_kv_gqa_gb300/csrc/plan.cpp"]


def profile_name(workload: str, cache: str = "bf16") -> str:
    return workload if cache == "bf16" else "%s_%s" % (workload, cache)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def causal_flops(case) -> int:
    """Multiply-add flops of a causal several-rows call: row i of a request with n rows and
    L keys sees L - n + i + 1 keys; each key costs 4 D flops per query head (scores, PV)."""
    import numpy as np
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    qo = case.qo_indptr.cpu().numpy().astype(np.int64)
    keys = 0
    for b in range(case.B):
        n, L = int(qo[b + 1] - qo[b]), int(lens[b])
        i = np.arange(n)
        keys += int(np.clip(L - n + i + 1, 0, L).sum())
    return 4 * keys * case.Hq * case.D


def _kernel_name(tc_rows: int, fp8: bool, q_len: int, D: int = 128) -> str:
    if tc_rows == 256:
        return "prefill_tc2_kernel (tcgen05, 256 rows/CTA)"
    if tc_rows == 128 and D == 256:
        return "prefill_tc256_kernel<%s> (tcgen05, 128 rows/CTA, 64-key tiles)" % ("fp8" if fp8 else "bf16")
    if tc_rows == 128:
        return "prefill_tc_kernel<%s> (tcgen05, 128 rows/CTA)" % ("fp8" if fp8 else "bf16")
    return "decode_split_kernel<%s%s> (one launch per call; split merge fused)" % (
        "fp8 cache" if fp8 else "bf16 cache", ", multi-row" if q_len > 1 else "")


def _roofline(args, case, q_len, fp8, tc_rows, peaks, gbs, mean_ms) -> dict:
    """The roofline of the call's one kernel.  The decode kernel: HBM bandwidth (algorithmic
    bytes over the measured copy bandwidth).  The tcgen05 kernels: whichever roof takes longer
    at its peak, the tensor cores (causal FLOPs over the measured bf16 peak) or HBM (a long
    table with few rows per group streams more bytes than the products take); the other roof's
    fraction rides along under "secondary".  DRAM traffic comes from the committed ncu summary
    of the same kernel and workload, taken on the current source, else null."""
    name = _kernel_name(tc_rows, fp8, q_len, case.D)
    if tc_rows:
        flops = causal_flops(case)
        tflops = flops / (mean_ms * 1e-3) / 1e12
        tensor = {"bound": "tensor", "achieved": round(tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                  "frac": round(tflops / peaks["bf16_tflops"], 4)}
        hbm = {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
               "frac": round(gbs / peaks["hbm_gbs"], 4)}
        t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = gbs * mean_ms * 1e-3 * 1e9 / (peaks["hbm_gbs"] * 1e9)  # algorithmic bytes at the HBM peak
        main, other = (hbm, tensor) if t_hbm > t_tensor else (tensor, hbm)
        return dict(main, traffic=None, kernel=name, peak_source=peaks["source"], secondary=other)
    traffic = profiled_traffic(profile_name(args.workload, args.cache)) if q_len == 1 else None
    return {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": name,
            "peak_source": peaks["source"]}


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    only if that summary was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_split_kernel_%s.md" % workload)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class L2Flush:
    """Evicts L2 before a timed step: rewrites a 2 x L2 buffer, then reads a second one,
    so that no dirty line of the flush is left to be written back inside the step."""

    def __init__(self, torch, dev, l2_bytes):
        self.torch = torch
        self.wbuf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def fill_(self, v):
        self.wbuf.fill_(v)
        self.torch.sum(self.rbuf, dim=0, keepdim=True, out=self.sink)


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of the timed GPU while the timed region runs.

    Two read-only sources: NVML, called through ctypes from a thread that polls every
    `interval_s` and stamps each sample with the host clock (so that only samples taken
    between the first and the last timed event are kept), and one `nvidia-smi --query-gpu`
    snapshot just before the first timed event and one just after the last.  Nothing is
    set: only query functions are called."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of the NVML API (nvmlClocksEventReason*)
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    REJECT = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "hw_power_brake_slowdown")

    def __init__(self, device_index: int, pci_bus_id: str = None, interval_s: float = 0.001):
        self.device_index = device_index
        self.pci_bus_id = pci_bus_id
        self.interval_s = interval_s
        self.samples = []  # (host time, sm MHz, reason bits, power W)
        self.snapshots = {}
        self.nvml = None
        self.handle = None
        self.max_mhz = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.window = None

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.pci_bus_id:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci_bus_id.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device_index), ctypes.byref(h)) == 0
        if not ok:
            return False
        self.nvml, self.handle = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        return True

    def _nvml_sample(self):
        import ctypes
        lib, h = self.nvml, self.handle
        mhz, bits, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        t = time.perf_counter()
        if lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(mhz)) != 0:
            return
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if get_reasons(h, ctypes.byref(bits)) != 0:
            bits.value = 0
        power = mw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else None
        self.samples.append((t, float(mhz.value), int(bits.value), power))

    def _poll(self):
        while not self.stop_flag.is_set():
            self._nvml_sample()
            time.sleep(self.interval_s)

    def snapshot(self, tag: str):
        """One nvidia-smi reading (read-only query), kept under `tag`."""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.device_index), "--query-gpu=" + self.QUERY,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            parts = [p.strip() for p in r.stdout.strip().splitlines()[0].split(",")]
        except (OSError, subprocess.SubprocessError, IndexError):
            return
        if len(parts) >= 9:
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            self.snapshots[tag] = {"sm_mhz": _num(parts[1]), "sm_max_mhz": _num(parts[2]), "power_w": _num(parts[3]),
                                   "reasons": [names[i] for i in range(4) if parts[5 + i].lower() == "active"]}

    def start(self):
        if self._nvml_open():
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()

    def mark(self, t0: float, t1: float):
        """The host-clock window of the timed region (first event recorded .. last event done)."""
        self.window = (t0, t1)

    def stop(self) -> dict:
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=5)
        if self.nvml is not None:
            self.nvml.nvmlShutdown()
        lo, hi = self.window if self.window else (-1e30, 1e30)
        inside = [s for s in self.samples if lo <= s[0] <= hi]
        sm = [s[1] for s in inside]
        reasons = sorted({name for s in inside for bit, name in self.REASON_BITS.items() if s[2] & bit})
        for snap in self.snapshots.values():
            reasons = sorted(set(reasons) | set(snap["reasons"]))
        power = [s[3] for s in inside if s[3] is not None]
        mx = self.max_mhz or max([s.get("sm_max_mhz") or 0 for s in self.snapshots.values()] or [0]) or None
        med = statistics.median(sm) if sm else None
        if med is None:  # no sample inside the region: the bracketing snapshots
            vals = [s["sm_mhz"] for s in self.snapshots.values() if s.get("sm_mhz")]
            med = statistics.median(vals) if vals else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": reasons,
                "samples_in_timed_region": len(inside), "sampler": "NVML every %.0f ms" % (self.interval_s * 1e3)
                if self.nvml is not None else "nvidia-smi snapshots only",
                "sm_mhz_min_max": [min(sm), max(sm)] if sm else None,
                "power_w_max": max(power) if power else None,
                "snapshots": self.snapshots,
                "rejected": any(r in self.REJECT for r in reasons)}


def _num(s):
    try:
        return float(s)
    except ValueError:
        return None


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("PKV_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, rank, world, local


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time: every rank contributes its value, all get the max."""
    if not dist:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processed bytes_per_rank in the slowest rank's time."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


def run_reference(args) -> None:
    """The oracle as it stands, timed on the host cores (one bounded sample per step)."""
    import numpy as np
    import oracle
    from workloads import algorithmic_bytes, make_case

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = make_case(args.workload)
    q, k, v, bt, sl = case.host_bits()
    cache = getattr(args, "cache", "bf16")
    if cache == "fp8":  # the oracle's own quantiser makes its fp8 cache
        k8, ks = oracle.quantize_pool(k)
        v8, vs = oracle.quantize_pool(v)
        run_rows = lambda sel: oracle.paged_decode_fp8(q, k8, v8, ks, vs, bt, sl, case.scale, select=sel)
    else:
        run_rows = lambda sel: oracle.paged_decode(q, k, v, bt, sl, case.scale, select=sel)
    # each step's sample is sized so that the whole run (warm-up and timed steps) stays within
    # a few minutes whatever the step count
    per_step = min(args.ref_seconds, _REFERENCE_RUN_SECONDS / (args.steps + args.warmup))
    rows, sample, cores = _reference_sample(case, per_step, _oracle_thread_rate(case, run_rows))
    one = lambda: run_rows(rows)
    ab = algorithmic_bytes(case, cache=cache)
    frac = len(rows) / (case.B * case.Hq)
    step_bytes = ab["total"] * frac
    for _ in range(args.warmup):
        one()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        t.append(time.perf_counter() - t0)
    sec = sum(t) / len(t)
    value = step_bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_block(case, args, plan=None),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# wall-clock budget of a whole `--impl reference` run (warm-up and timed steps together)
_REFERENCE_RUN_SECONDS = 150.0


def _oracle_thread_rate(case, run_rows) -> float:
    """fp64 flops a second of one oracle thread on this host: one row of the longest sequence,
    once untimed (a warm-up: the first pass over the inputs runs slower), then repeated for at
    least 20 ms."""
    import numpy as np
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    b = int(np.argmax(lens))
    flops = max(1, int(lens[b])) * case.D * 4.0
    run_rows([(b, 0)])
    n, t = 0, 0.0
    while t < 0.02 or n == 0:
        t0 = time.perf_counter()
        run_rows([(b, 0)])
        t += time.perf_counter() - t0
        n += 1
    return flops * n / t


def _reference_sample(case, seconds, rate):
    """Rows (b, h) for a bounded CPU sample: the first n of a head-major order (head 0 of every
    sequence, then head 1, ...), n as large as keeps one oracle pass within `seconds` on this
    host's cores at `rate` fp64 flops a second per thread (the oracle's threads take the rows by
    a fixed stride), and at least one row.  Where one row alone takes longer than `seconds`, the
    pass may take as long as that row (the other threads take rows beside it in the same time).
    Returns (rows, description, threads used)."""
    import numpy as np
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    order = [(b, h) for h in range(case.Hq) for b in range(case.B)]
    cost = np.array([lens[b] * case.D * 4.0 / rate for b, _ in order])
    cores = os.cpu_count() or 1
    budget = max(seconds, float(cost[0]))

    def pass_seconds(n):
        t = min(cores, n)
        return max(cost[i:n:t].sum() for i in range(t))

    lo, hi = 1, len(order)
    while lo < hi:  # the largest n whose pass fits (pass time grows with n)
        mid = (lo + hi + 1) // 2
        if pass_seconds(mid) <= budget:
            lo = mid
        else:
            hi = mid - 1
    rows = order[:lo]
    return rows, "%d of %d rows (head-major: head 0 of every sequence, then head 1, ...) per step" % (
        len(rows), case.B * case.Hq), min(cores, len(rows))


def _config_block(case, args, plan):
    lens = case.seq_lens.cpu().numpy()
    cfg = {"workload": args.workload, "cache": getattr(args, "cache", "bf16"), "q_len": getattr(args, "q_len", 1),
           "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D,
           "page_size": case.P, "num_pages": case.num_pages, "max_pages": case.max_pages,
           "seq_lens": {"min": int(lens.min()), "max": int(lens.max()), "sum": int(lens.sum())},
           "seed": case.meta["seed"], "l2": "flushed before every timed step: 2 x L2 bytes rewritten, then another 2 x L2 bytes read "
                 "(cold and clean L2 at the start of the step)"}
    if plan is not None:
        cfg.update({"num_splits": plan["num_splits"], "chunk_tokens": plan["chunk_tokens"],
                    "grid_blocks": plan["grid_blocks"], "blocks_per_sm": plan["blocks_per_sm"],
                    "rows_per_block": plan["rows_per_block"], "q_tiles": plan["q_tiles"]})
    return cfg


def _cpu_baseline(case, seconds: float, fp8=None) -> dict:
    """The oracle as it stands on the host cores, on a bounded sample of the workload.
    fp8: optional host (k8, v8, k_scale, v_scale) numpy arrays of an fp8 cache."""
    import oracle
    from workloads import algorithmic_bytes
    q, k, v, bt, sl = case.host_bits()
    if fp8:
        run_rows = lambda sel: oracle.paged_decode_fp8(q, *fp8, bt, sl, case.scale, select=sel)
    else:
        run_rows = lambda sel: oracle.paged_decode(q, k, v, bt, sl, case.scale, select=sel)
    rows, sample, cores = _reference_sample(case, 1.0, _oracle_thread_rate(case, run_rows))
    frac = len(rows) / (case.B * case.Hq)
    step_bytes = algorithmic_bytes(case, cache="fp8" if fp8 else "bf16")["total"] * frac
    n, t_total = 0, 0.0
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end or n == 0:
        t0 = time.perf_counter()
        run_rows(rows)
        t_total += time.perf_counter() - t0
        n += 1
    return {"value": round(step_bytes * n / t_total / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": "%s; %d passes in %.1f s" % (sample, n, t_total)}


def run_pkv(args) -> None:
    import torch
    import paged_kv_gqa_gb300 as pkv
    from workloads import algorithmic_bytes, make_case

    dist, rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load()

    q_len = getattr(args, "q_len", 1)
    if q_len > 1:  # several new tokens per sequence (a multi-token decode step)
        from workloads import CONFIGS, draw_seq_lens, make_prefill_case
        spec = CONFIGS[args.workload]
        kv_lens = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
        case = make_prefill_case(args.workload, [q_len] * spec["B"], kv_lens, device=dev)
    else:
        case = make_case(args.workload, device=dev)
    fp8 = args.cache == "fp8"
    pkv.set_prefill_tensor_cores({0: "off", 1: "auto", 2: "always", 3: "rows128"}[getattr(args, "tc", 1)])
    if getattr(args, "cluster_merge", None) is not None:
        pkv.set_cluster_merge(bool(args.cluster_merge))
    pools8 = None
    if fp8:  # quantise the pools on the device, then drop the bf16 copies
        pools8 = pkv.quantize_pool_fp8(case.k_cache, case.v_cache)
        torch.cuda.synchronize()
        case.k_cache = case.v_cache = None
        torch.cuda.empty_cache()
    ab = algorithmic_bytes(case, cache=args.cache)
    props = torch.cuda.get_device_properties(dev)
    if q_len > 1:
        total_q = int(case.q.shape[0])
        plan = pkv.prefill_plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, total_q, q_len,
                                      props.multi_processor_count, cache=args.cache)
        ws_bytes = plan["workspace_bytes"]
    else:
        plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, props.multi_processor_count,
                              cache=args.cache)
        ws_bytes = pkv.paged_decode_attn_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages,
                                                        cache=args.cache)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    rows_q = case.q.shape[0]
    out = torch.empty((rows_q, case.Hq, case.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows_q, case.Hq), dtype=torch.float32, device=dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = L2Flush(torch, dev, l2)
    stream = torch.cuda.current_stream(dev)
    launches_per_call = 1  # the split merge runs inside the decode kernel

    def call():
        if q_len > 1:
            kc, vc = (pools8[0], pools8[1]) if fp8 else (case.k_cache, case.v_cache)
            pkv.paged_prefill_attn(case.q, kc, vc, case.qo_indptr, case.block_table, case.seq_lens, q_len, case.scale,
                                   out, lse, ws, causal=True, stream=stream,
                                   fp8_scales=(pools8[2], pools8[3]) if fp8 else None)
        elif fp8:
            pkv.paged_decode_attn_fp8(case.q, *pools8, case.block_table, case.seq_lens, case.scale, out, lse, ws,
                                      stream=stream)
        else:
            pkv.paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale,
                                  out, lse, ws, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        call()
    torch.cuda.synchronize()
    if pkv.pkv_check_status(ws) != 0:
        raise RuntimeError("device status %d after warm-up" % pkv.pkv_check_status(ws))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local, _pci_bus_id(props))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.snapshot("before_first_event")
    sampler.start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    t_wall = t_wall1 - t_wall0
    sampler.mark(t_wall0, t_wall1)
    sampler.snapshot("after_last_event")
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    floor_us = _event_floor_us(torch, flush, stream)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = sum(step_ms) / len(step_ms)
    mean_ms = max_over_ranks(mean_ms, dist, dev)
    status = pkv.pkv_check_status(ws)

    # ---- end to end through the public API with host buffers -------------------
    e2e = None
    if not args.no_e2e and q_len == 1:
        e2e = _e2e(args, case, ab, pkv, torch, dev, stream, flush, plan, dist, pools8)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and q_len == 1:
        if fp8:
            hc = _host_case(case)
            cpu = _cpu_baseline(hc, args.cpu_seconds, fp8=tuple(t.cpu().numpy() for t in pools8))
        else:
            cpu = _cpu_baseline(case.to("cpu"), args.cpu_seconds)

    per_config = None
    if not args.no_per_config and q_len == 1 and world == 1:
        per_config = _per_config(args, pkv, torch, dev, stream, flush, props.multi_processor_count)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks = measured_peaks()
    gbs = weak_scaling_gbs(ab["total"], 1, mean_ms)
    # the kernel the call takes: the library's own plan (rows_per_block 128 or 256 = tensor cores)
    tc_rows = plan["rows_per_block"] if q_len > 1 and plan["rows_per_block"] >= 128 else 0
    roofline = _roofline(args, case, q_len, fp8, tc_rows, peaks, gbs, mean_ms)
    line = {
        "metric": METRIC, "value": round(gbs * world, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(mean_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled page pool)" + (
            "; K/V quantised on the device to e4m3 with per-(token, kv head) power-of-two scales" if fp8 else ""),
        "config": _config_block(case, args, plan),
        "us_per_call": round(mean_ms * 1e3, 3),
        "us_per_call_p10_p50_p90": [round(x * 1e3, 3) for x in _quantiles(step_ms)],
        "pct_of_measured_hbm": round(100 * gbs / peaks["hbm_gbs"], 2),
        "pct_of_nominal_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
        "algorithmic_bytes": ab["total"], "tail_bytes_touched": ab["tail_bytes"],
        "roofline": roofline,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clocks, "device_status": status, "wall_s_timed_region": round(t_wall, 3),
        "per_config": per_config,
        "event_floor_us": floor_us,
        "tensor": None if q_len == 1 else {
            "kernel": _kernel_name(tc_rows, fp8, q_len, case.D),
            "tflops": round(causal_flops(case) / (mean_ms * 1e-3) / 1e12, 2),
            "peak_tflops": peaks["bf16_tflops"],
            "frac": round(causal_flops(case) / (mean_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)},
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _per_config(args, pkv, torch, dev, stream, flush, sms):
    """Every decode workload on both caches, measured in this process after the headline:
    mean event time per call (L2 flushed before each), achieved GB/s of algorithmic bytes and
    the fraction of the measured copy bandwidth.  Each workload's inputs are built, timed and
    freed in turn."""
    from workloads import CONFIG_ORDER, algorithmic_bytes, make_case
    peak = measured_peaks()["hbm_gbs"]
    steps = max(20, min(args.steps, 200))
    res = {"steps": steps, "warmup": 3, "peak_gbs": peak, "bf16": {}, "fp8": {}}
    for name in CONFIG_ORDER:
        case = make_case(name, device=dev)
        pools8 = None
        for cache in ("bf16", "fp8"):
            if cache == "fp8":
                pools8 = pkv.quantize_pool_fp8(case.k_cache, case.v_cache)
                case.k_cache = case.v_cache = None
            ws = torch.zeros(pkv.paged_decode_attn_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.P,
                                                                  case.max_pages, cache=cache),
                             dtype=torch.uint8, device=dev)
            out = torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device=dev)
            if cache == "fp8":
                call = lambda: pkv.paged_decode_attn_fp8(case.q, *pools8, case.block_table, case.seq_lens,
                                                         case.scale, out, lse, ws, stream=stream)
            else:
                call = lambda: pkv.paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table,
                                                     case.seq_lens, case.scale, out, lse, ws, stream=stream)
            for _ in range(3):
                flush.fill_(1)
                call()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for s_, e_ in ev:
                flush.fill_(2)
                s_.record(stream)
                call()
                e_.record(stream)
            torch.cuda.synchronize()
            if pkv.pkv_check_status(ws) != 0:
                raise RuntimeError("device status %d on %s/%s" % (pkv.pkv_check_status(ws), name, cache))
            ms = sum(s_.elapsed_time(e_) for s_, e_ in ev) / steps
            ab = algorithmic_bytes(case, cache=cache)["total"]
            gbs = ab / (ms * 1e-3) / 1e9
            plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, cache=cache)
            res[cache][name] = {"us_per_call": round(ms * 1e3, 3), "gbs": round(gbs, 1),
                                "frac": round(gbs / peak, 4), "algorithmic_bytes": ab,
                                "num_splits": plan["num_splits"], "gpu_launches": steps}
            del ws, out, lse
        del case, pools8
        torch.cuda.empty_cache()
    return res


def _pci_bus_id(props):
    """The device's PCI address in NVML's form, from torch's device properties (None if absent)."""
    try:
        return "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except (AttributeError, TypeError):
        return None


def _event_floor_us(torch, flush, stream, n=200):
    """Mean time of a trivial kernel timed exactly like a step (events after the same flush):
    the launch and event overhead under every step time."""
    tiny = torch.zeros(16, device=flush.wbuf.device)
    for _ in range(10):
        flush.fill_(1)
        tiny.add_(1)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for s_, e_ in ev:
        flush.fill_(1)
        s_.record(stream)
        tiny.add_(1)
        e_.record(stream)
    torch.cuda.synchronize()
    return round(sum(s_.elapsed_time(e_) for s_, e_ in ev) / n * 1e3, 3)


def _quantiles(xs):
    s = sorted(xs)
    return [s[int(0.1 * (len(s) - 1))], s[int(0.5 * (len(s) - 1))], s[int(0.9 * (len(s) - 1))]]


def _host_case(case):
    """A host copy of a case whose bf16 pools were dropped (fp8 runs): q, table, lengths."""
    from workloads import Case
    c = Case(**case.__dict__)
    for n in ("q", "block_table", "seq_lens"):
        setattr(c, n, getattr(case, n).cpu())
    import torch
    c.k_cache = c.v_cache = torch.empty(0, dtype=torch.bfloat16)
    return c


def _e2e(args, case, ab, pkv, torch, dev, stream, flush, plan, dist, pools8=None):
    """Same metric, through the public call with host buffers: each step copies the
    step's inputs host -> device from pinned memory, runs the call, and reads the
    result back."""
    if pools8 is not None:
        host = {n: getattr(case, n).cpu().pin_memory() for n in ("q", "block_table", "seq_lens")}
        for n, t in zip(("k8", "v8", "ks", "vs"), pools8):
            host[n] = t.cpu().pin_memory()
    else:
        host = {n: getattr(case, n).cpu().pin_memory() for n in ("q", "k_cache", "v_cache", "block_table",
                                                                   "seq_lens")}
    devb = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    out_h = torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((case.B, case.Hq), dtype=torch.float32).pin_memory()
    out = torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(plan["workspace_bytes"], dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    steps = max(3, min(args.steps, args.e2e_steps))

    def step():
        for n in host:
            devb[n].copy_(host[n], non_blocking=True)
        if pools8 is not None:
            pkv.paged_decode_attn_fp8(devb["q"], devb["k8"], devb["v8"], devb["ks"], devb["vs"], devb["block_table"],
                                      devb["seq_lens"], case.scale, out, lse, ws, stream=stream)
        else:
            pkv.paged_decode_attn(devb["q"], devb["k_cache"], devb["v_cache"], devb["block_table"],
                                  devb["seq_lens"], case.scale, out, lse, ws, stream=stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in ev:
        flush.fill_(2)
        s.record(stream)
        step()
        e.record(stream)
    torch.cuda.synchronize()
    ms = sum(s.elapsed_time(e) for s, e in ev) / steps
    ms = max_over_ranks(ms, dist, dev)
    world = dist.get_world_size() if dist else 1
    return {"value": round(weak_scaling_gbs(ab["total"], world, ms), 3), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps}


def run_append(args) -> None:
    """The paged KV append (the cache write before a decode step) on the large-batch shape:
    B=256 sequences, Hkv=8, D=128, 64-key pages; each step writes one K row and one V row
    per (sequence, kv head) into the last slot of the sequence's last page."""
    import torch
    import paged_kv_gqa_gb300 as pkv
    from workloads import make_case

    if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
        return
    dev = torch.device("cuda", 0)
    case = make_case("bigpage", device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    kn = torch.randn(case.B, case.Hkv, case.D, generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn(case.B, case.Hkv, case.D, generator=g, device=dev).to(torch.bfloat16)
    pos = (case.seq_lens - 1).to(torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(torch, dev, 128 << 20)
    stream = torch.cuda.current_stream(dev)
    call = lambda: pkv.paged_kv_append(kn, vn, case.block_table, pos, case.k_cache, case.v_cache, status=status,
                                       stream=stream)
    for _ in range(args.warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s_, e_ in ev:
        flush.fill_(3)
        s_.record(stream)
        call()
        e_.record(stream)
    torch.cuda.synchronize()
    ms = sum(s_.elapsed_time(e_) for s_, e_ in ev) / len(ev)
    assert int(status.item()) == 0
    rows = case.B * case.Hkv
    moved = 2 * 2 * rows * case.D * 2 + case.B * 4 * 2  # K and V rows read and written, positions, table entries
    print(json.dumps({"metric": "paged KV append: us/call and achieved HBM GB/s", "value": round(moved / (ms * 1e-3) / 1e9, 2),
                      "unit": "GB/s", "us_per_call": round(ms * 1e3, 3), "steps": args.steps, "warmup": args.warmup,
                      "config": {"workload": "append", "B": case.B, "Hkv": case.Hkv, "D": case.D, "page_size": case.P},
                      "bytes_per_call": moved, "gpu_launches": args.steps}), flush=True)


def run_step(args) -> None:
    """One serving iteration on the batch workload: write each sequence's newest key and
    value (the last slot of its length), then decode over its keys.  Timed per step with
    CUDA events (L2 flushed before each step) four ways: serialised launches, programmatic
    dependent launch (PDL), the step captured in a CUDA graph, and a graph with PDL."""
    import torch
    import paged_kv_gqa_gb300 as pkv
    from workloads import algorithmic_bytes, make_case

    if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
        return
    dev = torch.device("cuda", 0)
    case = make_case("batch", device=dev)
    fp8 = args.cache == "fp8"
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    kn = torch.randn(case.B, case.Hkv, case.D, generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn(case.B, case.Hkv, case.D, generator=g, device=dev).to(torch.bfloat16)
    pos = (case.seq_lens - 1).to(torch.int32)
    pools = pkv.quantize_pool_fp8(case.k_cache, case.v_cache) if fp8 else None
    ws = torch.zeros(pkv.paged_decode_attn_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages,
                                                          cache=args.cache), dtype=torch.uint8, device=dev)
    out = torch.empty(case.B, case.Hq, case.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(case.B, case.Hq, dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev, getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    stream = torch.cuda.Stream(dev)

    def step():
        if fp8:
            pkv.paged_kv_append_fp8(kn, vn, case.block_table, pos, *pools, stream=stream)
            pkv.paged_decode_attn_fp8(case.q, *pools, case.block_table, case.seq_lens, case.scale, out, lse, ws,
                                      stream=stream)
        else:
            pkv.paged_kv_append(kn, vn, case.block_table, pos, case.k_cache, case.v_cache, stream=stream)
            pkv.paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale,
                                  out, lse, ws, stream=stream)

    def timed(run):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.fill_(1)
                run()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for s_, e_ in ev:
                flush.fill_(2)
                s_.record(stream)
                run()
                e_.record(stream)
        torch.cuda.synchronize()
        return sum(s_.elapsed_time(e_) for s_, e_ in ev) / len(ev) * 1e3

    res = {}
    for mode in ("serialised", "pdl", "graph", "graph+pdl"):
        pkv.set_programmatic_launch("pdl" in mode)
        if mode.startswith("graph"):
            with torch.cuda.stream(stream):
                step()  # first calls outside capture (attribute setup, tensor-map cache)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                step()
            res[mode] = timed(graph.replay)
        else:
            res[mode] = timed(step)
    pkv.set_programmatic_launch(False)
    assert pkv.pkv_check_status(ws) == 0
    ab = algorithmic_bytes(case, cache=args.cache)["total"] + 2 * 2 * case.B * case.Hkv * case.D * 2
    best = min(res.values())
    print(json.dumps({"metric": "decode step (KV append + paged decode attention): us/step", "value": round(best, 3),
                      "unit": "us", "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
                      "us_per_step": {k: round(v, 3) for k, v in res.items()},
                      "gb_per_s_best": round(ab / (best * 1e-6) / 1e9, 1),
                      "config": {"workload": "step", "base": "batch", "cache": args.cache, "B": case.B, "Hq": case.Hq,
                                 "Hkv": case.Hkv, "D": case.D, "page_size": case.P,
                                 "l2": "flushed before every timed step (write 2 x L2, read another 2 x L2)"},
                      "gpu_launches": 2 * args.steps * 4}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long",
                    choices=["tiny", "batch", "ragged", "long", "bigpage", "bigpage_g16", "append", "step"])
    ap.add_argument("--cache", default="bf16", choices=["bf16", "fp8"])
    ap.add_argument("--q-len", type=int, default=1,
                    help="new tokens per sequence (causal multi-token step); 1 = decode")
    ap.add_argument("--cluster-merge", type=int, default=None, choices=[0, 1],
                    help="decode split merge through a thread-block cluster (pkv_set_cluster_merge); "
                         "default: the library's setting")
    ap.add_argument("--tc", type=int, default=1, choices=[0, 1, 2, 3],
                    help="several-rows calls: 0 = mma.sync kernel, 1 = library routing (pkv_set_prefill_tensor_cores "
                         "auto), 2 = tensor-core kernel wherever it applies (256 rows per CTA where the group has "
                         "them), 3 = tensor-core kernel with 128 rows per CTA")
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the table of every decode workload on both caches after the headline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=1.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload == "append":
        run_append(args)
    elif args.workload == "step":
        run_step(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
