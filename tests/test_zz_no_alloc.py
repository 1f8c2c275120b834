"""The allocation-free decode entry point, paged_decode_attn_static_scratch.

It serves callers that cannot allocate device memory when they run attention
(a serving loop whose memory pool is frozen at start-up, a plugin handed only
one step's tensors): the split partials live in the library's own fixed device
array instead of a caller workspace.  These tests call it through the C ABI and
hold it to the workspace entry point's results, on two calls in a row.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, compare_with_oracle
from workloads import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def _call_static(lib, c, out, lse, status):
    V = ctypes.c_void_p
    return lib.paged_decode_attn_static_scratch(
        V(c.q.data_ptr()), V(c.k_cache.data_ptr()), V(c.v_cache.data_ptr()), V(c.block_table.data_ptr()),
        V(c.seq_lens.data_ptr()), c.B, c.Hq, c.Hkv, c.D, c.P, c.num_pages, c.max_pages, ctypes.c_float(c.scale),
        V(out.data_ptr()), V(lse.data_ptr()), V(status.data_ptr()),
        V(torch.cuda.current_stream().cuda_stream))


def _reference(c):
    ws = torch.zeros(pkv.paged_decode_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.B, c.Hq), dtype=torch.float32, device="cuda")
    pkv.paged_decode_attn(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale, out, lse, ws)
    assert pkv.pkv_check_status(ws) == 0
    return out, lse


def test_static_scratch_matches_workspace_entry_point_twice(lib):
    # Two shapes back to back, each planned with several splits, so the shared
    # scratch really carries partials and the second call sees the first one's leftovers.
    # Both entry points take the same plan and the same kernel, so their results agree
    # bit for bit; the first shape is also held to the oracle.
    cases = [
        make_case(dict(B=3, Hq=32, Hkv=8, D=128, P=16, lens=("fixed", 1), seed=31), seq_lens=[5000, 17, 1200]),
        make_case(dict(B=2, Hq=32, Hkv=2, D=256, P=64, lens=("fixed", 1), seed=32), seq_lens=[3000, 700]),
        # G = 32 at D = 256: two query tiles per group (one merge counter per tile)
        make_case(dict(B=2, Hq=64, Hkv=2, D=256, P=16, lens=("fixed", 1), seed=35), seq_lens=[2600, 90]),
    ]
    for n, c in enumerate(cases):
        c = c.to("cuda")
        plan = pkv.plan_query(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages,
                              torch.cuda.get_device_properties(0).multi_processor_count)
        assert plan["num_splits"] > 1
        assert plan["q_tiles"] == (2 if n == 2 else 1), plan
        ref_out, ref_lse = _reference(c)
        for _ in range(2):
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
            assert _call_static(lib, c, out, lse, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        if n != 1:
            eo, el = compare_with_oracle(c, out, lse)
            assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_static_scratch_clears_status_between_calls(lib):
    bad = make_case(dict(B=2, Hq=16, Hkv=4, D=128, P=16, lens=("fixed", 1), seed=33), seq_lens=[900, 40])
    bad.block_table[0, 2] = bad.num_pages + 7
    good = make_case(dict(B=2, Hq=16, Hkv=4, D=128, P=16, lens=("fixed", 1), seed=34), seq_lens=[900, 40])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c, want in ((bad, -6), (good, 0)):
        c = c.to("cuda")
        out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((c.B, c.Hq), dtype=torch.float32, device="cuda")
        assert _call_static(lib, c, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == want


def test_static_scratch_rejects_shapes_beyond_its_size(lib):
    # 64 sequences x 64 query heads of D=256 over 131072 keys need far more than 32 MiB of partials.
    V = ctypes.c_void_p
    plan = pkv.plan_query(64, 64, 2, 256, 16, 8192, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["workspace_bytes"] > 32 << 20
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = V(dummy.data_ptr())
    st = lib.paged_decode_attn_static_scratch(p, p, p, p, p, 64, 64, 2, 256, 16, 8192 * 64, 8192,
                                              ctypes.c_float(0.0625), p, None, None,
                                              V(torch.cuda.current_stream().cuda_stream))
    assert st == -4
