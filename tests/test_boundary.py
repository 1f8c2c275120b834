"""The C-ABI boundary without a GPU: the library loads, exports every declared
symbol, rejects bad arguments before touching CUDA, and plans deterministically."""
import ctypes
import os
import re

import pytest

import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    assert sorted(pkv.EXPORTED_SYMBOLS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_no_internal_symbols_leak():
    _build.build()
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {n for n in exported if n.startswith(("pkv", "paged_decode", "paged_kv", "paged_prefill", "split_kv"))}
    assert ours == set(_declared())


def test_status_strings(lib):
    for code, name in pkv.STATUS.items():
        assert pkv.status_string(code) == name
    assert pkv.status_string(12345) == "PKV_UNKNOWN_STATUS"
    assert lib.pkv_version() >= 100


def _call_decode(lib, q=0x1000, k=0x2000, v=0x3000, bt=0x4000, sl=0x5000, B=2, Hq=8, Hkv=2, D=128, P=16,
                 num_pages=64, max_pages=8, scale=0.125, out=0x6000, lse=0x7000, ws=0x8000, ws_bytes=1 << 20,
                 splits=0):
    """Fake (never dereferenced) pointers: every case below must be rejected on the host."""
    V = ctypes.c_void_p
    return lib.paged_decode_attn_ex(V(q), V(k), V(v), V(bt), V(sl), B, Hq, Hkv, D, P, num_pages, max_pages,
                                    ctypes.c_float(scale), V(out), V(lse), V(ws), ws_bytes, splits, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(bt=0), -1), (dict(sl=0), -1), (dict(out=0), -1),
    (dict(ws=0), -1), (dict(Hq=0), -1), (dict(Hkv=0), -1), (dict(Hq=6, Hkv=4), -1), (dict(B=-1), -1),
    (dict(num_pages=0), -1), (dict(max_pages=0), -1), (dict(splits=-2), -1), (dict(scale=float("nan")), -1),
    (dict(D=96), -2), (dict(D=32), -2), (dict(P=12), -2), (dict(P=4), -2), (dict(P=512), -2),
    (dict(Hq=66, Hkv=1), -2),
    (dict(q=0x1008), -3), (dict(k=0x2004), -3), (dict(bt=0x4002), -3), (dict(lse=0x7001), -3), (dict(ws=0x8008), -3),
])
def test_host_rejects_bad_arguments(lib, kw, status):
    assert _call_decode(lib, **kw) == status


def test_batch_zero_is_a_noop(lib):
    assert _call_decode(lib, B=0, q=0, k=0, v=0) == 0


def test_merge_rejects_bad_arguments(lib):
    V = ctypes.c_void_p
    assert lib.split_kv_merge(V(0x1000), V(0x2000), 0, 1, 1, 128, V(0x3000), None, None) == -1
    assert lib.split_kv_merge(V(0x1000), V(0x2000), 2, 1, 1, 96, V(0x3000), None, None) == -2
    assert lib.split_kv_merge(V(0x1004), V(0x2000), 2, 1, 1, 128, V(0x3000), None, None) == -3
    assert lib.split_kv_merge(V(0), V(0x2000), 2, 1, 1, 128, V(0x3000), None, None) == -1
    assert lib.split_kv_merge(V(0x1000), V(0x2000), 2, 0, 1, 128, V(0x3000), None, None) == 0


def test_status_calls_reject_null(lib):
    v = ctypes.c_int(0)
    assert lib.pkv_check_status(None, None, ctypes.byref(v)) == -1
    assert lib.pkv_reset_status(None, None) == -1
    assert lib.pkv_selftest_wait_timeout(None, 10, None) == -1
    assert lib.pkv_selftest_wait_timeout(ctypes.c_void_p(0x1000), 0, None) == -1


# ----------------------------------------------------------------- planner (pure host function)

WORKLOADS = {
    "tiny": (1, 8, 2, 64, 16, 16),
    "batch": (8, 32, 8, 128, 16, 256),
    "ragged": (64, 32, 8, 128, 16, 2048),
    "long": (4, 64, 8, 128, 16, 8192),
    "bigpage": (256, 32, 8, 128, 64, 32),
    "bigpage_g16": (256, 32, 2, 256, 64, 32),
}


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("sms", [148, 152, 160])
def test_plan_invariants(lib, name, sms, cache):
    B, Hq, Hkv, D, P, max_pages = WORKLOADS[name]
    plan = pkv.plan_query(B, Hq, Hkv, D, P, max_pages, sms, cache=cache)
    max_tokens = max_pages * P
    assert plan["chunk_tokens"] % plan["stage_tokens"] == 0
    assert plan["num_splits"] * plan["chunk_tokens"] >= max_tokens
    assert (plan["num_splits"] - 1) * plan["chunk_tokens"] < max_tokens
    assert plan["smem_bytes"] <= 232448
    assert plan["grid_blocks"] == plan["num_splits"] * Hkv * B
    # 2-8 splits on a grid of one wave merge inside a cluster (on by default), more through the workspace
    if plan["num_splits"] == 1:
        assert plan["merge_needed"] == 0
    elif plan["merge_needed"] == 2:
        assert plan["num_splits"] <= 8 and plan["grid_blocks"] <= sms * plan["blocks_per_sm"], plan
    else:
        assert plan["merge_needed"] == 1
    # cache bytes of one split (K and V; fp8: codes and scales) stay bounded (<= 2 MiB) so no
    # split becomes a straggler
    token_bytes = 4 * D if cache == "bf16" else 2 * D + 8
    assert plan["chunk_tokens"] * token_bytes <= (2 << 20) or plan["num_splits"] == 1
    if plan["num_splits"] > 1:
        pad = lambda x: (x + 255) // 256 * 256
        ws = 256 + pad(B * Hkv * 4) + pad(plan["num_splits"] * B * Hq * 4) + plan["num_splits"] * B * Hq * D * 4
        assert plan["workspace_bytes"] == ws
    else:
        assert plan["workspace_bytes"] == 256
    # a pure function of (shape, SM count, cache type)
    assert pkv.plan_query(B, Hq, Hkv, D, P, max_pages, sms, cache=cache) == plan


def test_plan_splits_long_context_and_not_big_batches(lib):
    assert pkv.plan_query(4, 64, 8, 128, 16, 8192, 152)["num_splits"] >= 32
    assert pkv.plan_query(256, 32, 8, 128, 64, 32, 152)["num_splits"] == 1
    # a small batch is split into about one wave of blocks
    p = pkv.plan_query(8, 32, 8, 128, 16, 247, 152)
    assert 3 <= p["num_splits"] <= 8 and p["grid_blocks"] <= 2 * 2 * 152


def test_plan_forced_splits(lib):
    for s in (1, 2, 3, 7, 64):
        plan = pkv.plan_query(8, 32, 8, 128, 16, 256, 152, s)
        assert plan["num_splits"] == s
    # clamped to one split per stage
    assert pkv.plan_query(1, 8, 2, 64, 16, 2, 152, 1000)["num_splits"] == 1
    with pytest.raises(pkv.PkvError):
        pkv.plan_query(1, 8, 2, 64, 16, 2, 152, -1)


def test_append_rejects_bad_arguments(lib):
    V = ctypes.c_void_p

    def call(kn=0x1000, vn=0x2000, bt=0x3000, pos=0x4000, B=2, Hkv=2, D=128, P=16, npg=8, mp=4,
             kc=0x5000, vc=0x6000, st=None):
        return lib.paged_kv_append(V(kn), V(vn), V(bt), V(pos), B, Hkv, D, P, npg, mp, V(kc), V(vc),
                                   V(st) if st else None, None)

    assert call(kn=0) == -1 and call(kc=0) == -1 and call(npg=0) == -1 and call(Hkv=0) == -1
    assert call(D=96) == -2 and call(P=12) == -2
    assert call(vn=0x2008) == -3 and call(pos=0x4004) == -3 and call(st=0x7002) == -3
    assert call(B=0, kn=0, vn=0) == 0


def test_fp8_decode_rejects_bad_arguments(lib):
    V = ctypes.c_void_p

    def call(ks=0x9000, vs=0xA000, q=0x1000, k=0x2000, B=2, D=128, P=16, splits=0):
        return lib.paged_decode_attn_fp8(V(q), V(k), V(0x3000), V(ks), V(vs), V(0x4000), V(0x5000), B, 8, 2, D, P,
                                         64, 8, ctypes.c_float(0.125), V(0x6000), V(0x7000), V(0x8000), 1 << 20,
                                         splits, None)

    assert call(ks=0) == -1 and call(vs=0) == -1 and call(q=0) == -1 and call(splits=-1) == -1
    assert call(ks=0x9004) == -3 and call(vs=0xA008) == -3 and call(k=0x2001) == -3
    assert call(D=96) == -2 and call(P=4) == -2
    assert call(B=0, q=0, k=0, ks=0, vs=0) == 0


def test_fp8_append_rejects_bad_arguments(lib):
    V = ctypes.c_void_p

    def call(ks=0x7000, vs=0x8000, kn=0x1000, kc=0x5000, B=2, D=128):
        return lib.paged_kv_append_fp8(V(kn), V(0x2000), V(0x3000), V(0x4000), B, 2, D, 16, 8, 4, V(kc), V(0x6000),
                                       V(ks), V(vs), None, None)

    assert call(ks=0) == -1 and call(vs=0) == -1 and call(kn=0) == -1
    assert call(ks=0x7004) == -3 and call(kc=0x5008) == -3
    assert call(D=32) == -2
    assert call(B=0, kn=0, ks=0, vs=0) == 0


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_residency_and_ring_per_cache(lib, name):
    # one head tile (G <= 8): three blocks per SM for either cache (bf16 with a 2-deep
    # ring of 16-key stages, fp8 with a 2-deep ring of 32-key stages at D = 128, 4-deep at
    # D = 64); otherwise two; D = 256: one bf16 block (3-deep ring), two fp8 blocks
    # (3-deep) up to 16 heads per group
    B, Hq, Hkv, D, P, max_pages = WORKLOADS[name]
    b = pkv.plan_query(B, Hq, Hkv, D, P, max_pages, 152)
    f = pkv.plan_query(B, Hq, Hkv, D, P, max_pages, 152, cache="fp8")
    G = Hq // Hkv
    if D == 256:
        assert (b["blocks_per_sm"], b["ring_stages"]) == (1, 3)
        assert (f["blocks_per_sm"], f["ring_stages"]) == ((2, 3) if G <= 16 else (1, 6))
    else:
        assert (b["blocks_per_sm"], b["ring_stages"]) == ((3, 2) if G <= 8 else (2, 3))
        if G <= 8:
            want = (3, 2, 32) if D == 128 else (3, 4, 32)
        else:
            want = (2, 6, 16 if D == 128 else 32)
        assert (f["blocks_per_sm"], f["ring_stages"], f["stage_tokens"]) == want
    for p in (b, f):
        assert p["blocks_per_sm"] * (p["smem_bytes"] + 1024) <= 233472
    assert f["warps"] == b["warps"]


def test_plan_rejects_unknown_kv_dtype(lib):
    plan = pkv.PkvPlan()
    assert lib.pkv_plan_query_kv(8, 32, 8, 128, 16, 64, 152, 0, 2, ctypes.byref(plan)) == -1
    n = ctypes.c_size_t(0)
    assert lib.paged_decode_attn_workspace_size_kv(8, 32, 8, 128, 16, 64, 0, 0, 7, ctypes.byref(n)) == -1


def test_tensor_core_routing_modes(lib):
    # the process-wide switch: each mode round-trips, unknown ones are refused on both sides
    old = pkv.set_prefill_tensor_cores("auto")
    try:
        for mode in ("off", "always", "rows128", "auto"):
            pkv.set_prefill_tensor_cores(mode)
        assert pkv.set_prefill_tensor_cores("rows128") == "auto"
        assert pkv.set_prefill_tensor_cores(True) == "rows128"
        assert pkv.set_prefill_tensor_cores(False) == "auto"
        assert pkv.set_prefill_tensor_cores("auto") == "off"
        with pytest.raises(ValueError):
            pkv.set_prefill_tensor_cores("fast")
        assert lib.pkv_set_prefill_tensor_cores(7) == -1
        assert pkv.set_prefill_tensor_cores("auto") == "auto"  # the refused call changed nothing
    finally:
        pkv.set_prefill_tensor_cores(old)


def _tc_splits(B, Hkv, G, max_pages, P, max_q, num_splits, rows, sms):
    """The tensor-core split plan restated: fewer groups than SMs -> the count that minimises
    waves x (tiles per CTA + 16), else chunks of at most 64 key tiles; num_splits > 0 forces
    the count."""
    max_tiles = max(1, -(-max_pages * P // 128))
    groups = B * Hkv * -(-max_q * G // rows)
    if num_splits > 0:
        s = num_splits
    elif groups < sms:
        costs = [(-(-groups * n // sms) * (-(-max_tiles // n) + 16), n)
                 for n in range(1, max(1, min(max_tiles, 4 * sms // groups)) + 1)]
        s = min(costs)[1]
    else:
        s = -(-max_tiles // 64)
    chunk = -(-max_tiles // min(max(s, 1), max_tiles, 65535))
    return -(-max_tiles // chunk)


@pytest.mark.parametrize("B,max_q,max_pages,num_splits,sms", [
    (4, 128, 1024, 0, 152),    # 64 groups of 256 rows: 2 splits; 128 groups of 128 rows: 1
    (1, 32, 8192, 0, 152),     # 8 groups: 19 splits (one wave)
    (64, 64, 2048, 0, 152),    # 512 groups: 64-tile chunks of a 256-tile table, 4 splits
    (4, 128, 1024, 3, 152),    # forced
    (8, 512, 256, 0, 152),     # 512 groups, 32 tiles: no split
    (4, 16, 1024, 0, 152),     # 64 rows per group: the 128-row kernel may take it, 32 groups -> 9 splits
    (4, 64, 8192, 0, 152),     # the long workload's shape at 16 new tokens: 32 groups -> 9 splits
])
def test_prefill_workspace_covers_tensor_core_splits(lib, B, max_q, max_pages, num_splits, sms):
    # bf16, D = 128, G = 4: the tensor-core kernels may take the call, so the plan's workspace
    # holds their split partials: splits x rows x (D + 1) floats plus a counter per group
    Hq, Hkv, D, P = 32, 8, 128, 16
    total_q = B * max_q
    plan = pkv.prefill_plan_query(B, Hq, Hkv, D, P, max_pages, total_q, max_q, sms, num_splits=num_splits)
    rows = total_q * Hq
    need = 0
    for cta_rows in (128, 256):
        s = _tc_splits(B, Hkv, Hq // Hkv, max_pages, P, max_q, num_splits, cta_rows, sms)
        if s > 1:
            need = max(need, s * rows * (D + 1) * 4)
    assert plan["workspace_bytes"] >= need
    if num_splits == 0 and (B, max_q, max_pages) == (1, 32, 8192):
        assert need == 19 * rows * (D + 1) * 4  # 8 groups of 1024 tiles: 19 splits fill one wave
    if num_splits == 0 and (B, max_q, max_pages) == (4, 64, 8192):
        # 32 groups of 1024 tiles: 4 splits (one wave of 128 CTAs, 1 x (256 + 16)) lose to 9 (two
        # waves of 288 CTAs, 2 x (114 + 16)), measured 434 vs 401 us on the long workload
        assert need == 9 * rows * (D + 1) * 4
    # the fp8 cache never takes the tensor-core kernels: its plan is the mma.sync kernel's alone
    fp8 = pkv.prefill_plan_query(B, Hq, Hkv, D, P, max_pages, total_q, max_q, sms, num_splits=num_splits, cache="fp8")
    assert fp8["workspace_bytes"] <= plan["workspace_bytes"]


@pytest.mark.parametrize("shape,cache,expect", [
    # (B, Hq, Hkv, D, P, max_pages, max_q): rows per group = max_q * Hq / Hkv
    ((8, 32, 8, 128, 16, 247, 512), "bf16", {"off": 0, "auto": 256, "always": 256, "rows128": 128}),
    ((8, 32, 8, 128, 16, 247, 512), "fp8", {"off": 0, "auto": 128, "always": 128, "rows128": 128}),
    ((4, 64, 8, 128, 16, 8192, 8), "bf16", {"off": 0, "auto": 128, "always": 128, "rows128": 128}),  # 64 rows, 128K keys
    ((4, 64, 8, 128, 16, 8192, 8), "fp8", {"off": 0, "auto": 128, "always": 128, "rows128": 128}),
    ((4, 64, 8, 128, 16, 256, 8), "bf16", {"off": 0, "auto": 0, "always": 128, "rows128": 128}),     # 64 rows, 4K keys
    ((4, 64, 8, 128, 16, 8192, 4), "bf16", {"off": 0, "auto": 0, "always": 0, "rows128": 0}),         # 32 rows: one block
    ((1, 8, 1, 128, 16, 2, 32), "bf16", {"off": 0, "auto": 128, "always": 256, "rows128": 128}),      # 256 rows, 1 CTA
    ((2, 16, 2, 64, 16, 8192, 64), "bf16", {"off": 0, "auto": 0, "always": 0, "rows128": 0}),         # D = 64
])
def test_prefill_plan_names_the_kernel_the_routing_takes(lib, shape, cache, expect):
    # the plan of a several-rows call under each routing: rows_per_block 128 / 256 = the tensor-core
    # kernels (with their key splits and grid), else the mma.sync kernel's plan (<= 32 rows per block)
    B, Hq, Hkv, D, P, max_pages, max_q = shape
    total_q = B * max_q
    old = pkv.set_prefill_tensor_cores("auto")
    try:
        ws = set()
        for mode, rows in expect.items():
            pkv.set_prefill_tensor_cores(mode)
            plan = pkv.prefill_plan_query(B, Hq, Hkv, D, P, max_pages, total_q, max_q, 152, cache=cache)
            ws.add(plan["workspace_bytes"])
            if rows == 0:
                assert plan["rows_per_block"] <= 32, (mode, plan)
                continue
            assert plan["rows_per_block"] == rows, (mode, plan)
            s = _tc_splits(B, Hkv, Hq // Hkv, max_pages, P, max_q, 0, rows, 152)
            q_tiles = -(-max_q * (Hq // Hkv) // rows)
            assert plan["num_splits"] == s and plan["q_tiles"] == q_tiles
            assert plan["grid_blocks"] == B * Hkv * q_tiles * s and plan["merge_needed"] == (s > 1)
            assert plan["blocks_per_sm"] == 1 and plan["stage_tokens"] == 128
        assert len(ws) == 1  # the workspace covers every routing, so it does not depend on the mode
    finally:
        pkv.set_prefill_tensor_cores(old)


def _call_prefill(lib, fp8=False, q=0x1000, k=0x2000, v=0x3000, qo=0x9000, bt=0x4000, sl=0x5000, B=2, Hq=8, Hkv=2,
                  D=128, P=16, num_pages=64, max_pages=8, total_q=6, max_q_len=4, causal=1, scale=0.125, out=0x6000,
                  lse=0x7000, ws=0x8000, ws_bytes=1 << 20, splits=0, ks=0xa000, vs=0xb000):
    """Fake (never dereferenced) pointers: every case below must be rejected on the host."""
    V = ctypes.c_void_p
    if fp8:
        return lib.paged_prefill_attn_fp8(V(q), V(k), V(v), V(ks), V(vs), V(qo), V(bt), V(sl), B, Hq, Hkv, D, P,
                                          num_pages, max_pages, total_q, max_q_len, causal, ctypes.c_float(scale),
                                          V(out), V(lse), V(ws), ws_bytes, splits, None)
    return lib.paged_prefill_attn(V(q), V(k), V(v), V(qo), V(bt), V(sl), B, Hq, Hkv, D, P, num_pages, max_pages,
                                  total_q, max_q_len, causal, ctypes.c_float(scale), V(out), V(lse), V(ws), ws_bytes,
                                  splits, None)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(qo=0), -1), (dict(total_q=-1), -1), (dict(max_q_len=0), -1), (dict(causal=2), -1),
    (dict(q=0), -1), (dict(bt=0), -1), (dict(Hq=6, Hkv=4), -1), (dict(scale=float("inf")), -1),
    (dict(D=96), -2), (dict(P=12), -2),
    (dict(qo=0x9004), -3), (dict(q=0x1008), -3), (dict(out=0x6008), -3),
])
def test_prefill_host_rejects_bad_arguments(lib, fp8, kw, status):
    # the several-rows entry points check their row ranges and pointers on the host, before any launch
    assert _call_prefill(lib, fp8=fp8, **kw) == status


def test_prefill_fp8_scales_are_checked(lib):
    assert _call_prefill(lib, fp8=True, ks=0) == -1
    assert _call_prefill(lib, fp8=True, vs=0) == -1
    assert _call_prefill(lib, fp8=True, ks=0xa004) == -3


def test_prefill_without_rows_is_a_noop(lib):
    assert _call_prefill(lib, total_q=0, q=0, k=0, v=0) == 0
    assert _call_prefill(lib, fp8=True, total_q=0, q=0, k=0, v=0) == 0


def test_static_scratch_rejects_bad_arguments_before_touching_cuda(lib):
    # Without a GPU any CUDA call would fail (PKV_ERR_CUDA), so a misaligned or malformed call
    # that returns its own status was rejected before the scratch array was touched.
    V = ctypes.c_void_p

    def call(q=0x1000, bt=0x4000, out=0x6000, lse=0x7000, status=0x9000, B=2, D=128, num_pages=64, scale=0.125):
        return lib.paged_decode_attn_static_scratch(V(q), V(0x2000), V(0x3000), V(bt), V(0x5000), B, 8, 2, D, 16,
                                                    num_pages, 8, ctypes.c_float(scale), V(out), V(lse), V(status),
                                                    None)
    assert call(q=0x1008) == -3
    assert call(bt=0x4004) == -3
    assert call(lse=0x7002) == -3
    assert call(status=0x9002) == -3
    assert call(out=0) == -1
    assert call(num_pages=0) == -1
    assert call(num_pages=1 << 27) == -1  # num_pages * page_size past int32
    assert call(scale=float("inf")) == -1
    assert call(D=96) == -2
    assert call(B=0, q=0) == 0


def test_plan_reports_cluster_merge(lib):
    # decode with 2-8 splits merges inside a cluster; more splits, one split, several rows per
    # sequence, or the switch off: the workspace merge (or none)
    prev = pkv.set_cluster_merge(True)
    assert prev is True  # on at load
    try:
        for S in range(2, 9):
            assert pkv.plan_query(4, 32, 8, 128, 16, 256, 152, num_splits=S)["merge_needed"] == 2
            assert pkv.plan_query(4, 32, 8, 128, 16, 256, 152, num_splits=S, cache="fp8")["merge_needed"] == 2
        # more blocks than one wave (8 x 8 x 8 on 152 SMs x 3): the workspace merge
        assert pkv.plan_query(8, 32, 8, 128, 16, 256, 152, num_splits=8)["merge_needed"] == 1
        assert pkv.plan_query(8, 32, 8, 128, 16, 256, 152, num_splits=9)["merge_needed"] == 1
        # G = 32 at D = 128: split 0's ring cannot hold 5 partials of 32 rows beside its combine buffer
        assert pkv.plan_query(2, 64, 2, 128, 16, 256, 152, num_splits=6)["merge_needed"] == 1
        assert pkv.plan_query(2, 32, 2, 128, 16, 256, 152, num_splits=6)["merge_needed"] == 2
        assert pkv.plan_query(4, 64, 8, 128, 16, 8192, 152)["merge_needed"] == 1      # long: 42 splits
        assert pkv.plan_query(256, 32, 8, 128, 64, 32, 152)["merge_needed"] == 0      # big pages: one split
        assert pkv.plan_query(8, 32, 8, 128, 16, 256, 152)["merge_needed"] == 2       # batch: 5 splits
        assert pkv.prefill_plan_query(8, 32, 8, 128, 16, 256, 32, 4, 152, num_splits=4)["merge_needed"] == 1
        assert pkv.set_cluster_merge(False) is True
        assert pkv.plan_query(8, 32, 8, 128, 16, 256, 152, num_splits=4)["merge_needed"] == 1
    finally:
        pkv.set_cluster_merge(prev)


def test_prefill_plan_at_head_dim_256(lib):
    # D = 256: groups of more than 32 rows may take the 128-row tensor-core kernel of 64-key tiles
    # (on the fp8 cache its instantiation with converter warps)
    try:
        pkv.set_prefill_tensor_cores("auto")
        p = pkv.prefill_plan_query(256, 32, 2, 256, 64, 32, 256 * 8, 8, 152)  # 128 rows per group
        assert p["rows_per_block"] == 128 and p["stage_tokens"] == 64 and p["warps"] == 7
        # workspace: the status word, counters and partials of every split the kernel can take
        for splits in (0, 4):
            q = pkv.prefill_plan_query(2, 16, 2, 256, 16, 600, 18, 9, 152, num_splits=splits)
            assert q["rows_per_block"] == 128
            if q["num_splits"] > 1:
                assert q["workspace_bytes"] >= q["num_splits"] * 18 * 16 * 256 * 4
        p8 = pkv.prefill_plan_query(256, 32, 2, 256, 64, 32, 256 * 8, 8, 152, cache="fp8")
        assert p8["rows_per_block"] == 128 and p8["stage_tokens"] == 64 and p8["warps"] == 11, p8
        assert p8["smem_bytes"] <= 232448 and p8["ring_stages"] == 1
        pkv.set_prefill_tensor_cores("off")
        assert pkv.prefill_plan_query(256, 32, 2, 256, 64, 32, 256 * 8, 8, 152)["rows_per_block"] <= 32
    finally:
        pkv.set_prefill_tensor_cores("auto")


def test_head_dim_256_blocks_take_at_most_16_rows(lib):
    # At D = 256 a decode block serves at most 16 (token, head) rows: a group of 32 query heads, or a
    # 2-token step of a 16-head group, takes two query tiles (the 32-row variant would spill)
    for cache in ("bf16", "fp8"):
        p = pkv.plan_query(2, 64, 2, 256, 16, 100, 152, cache=cache)  # G = 32
        assert p["rows_per_block"] == 16 and p["q_tiles"] == 2, p
        assert p["grid_blocks"] == 2 * 2 * 2 * p["num_splits"]
        if p["num_splits"] > 1:  # the split counters cover both query tiles of every group
            pad = lambda x: (x + 255) // 256 * 256
            S = p["num_splits"]
            assert p["workspace_bytes"] == 256 + pad(2 * 2 * 2 * 4) + pad(S * 2 * 64 * 4) + S * 2 * 64 * 256 * 4
        q = pkv.prefill_plan_query(256, 32, 2, 256, 64, 32, 256 * 2, 2, 152, cache=cache)  # 32 rows per group
        assert q["rows_per_block"] == 16 and q["q_tiles"] == 2, q
    # D = 128 keeps 32-row blocks
    assert pkv.plan_query(2, 64, 2, 128, 16, 100, 152)["rows_per_block"] == 32
