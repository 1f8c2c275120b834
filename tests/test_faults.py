"""Failure detection on the GPU without a GPU fault.

Bad device data (a page id out of range, a length past the table) is skipped by
the kernel and reported through the workspace status word; a stalled copy ends
in a bounded wait that reports PKV_ERR_DEVICE_TIMEOUT.  Nothing here traps,
faults or hangs the device, and the context stays usable afterwards.
"""
import pytest
import torch

import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, compare_with_oracle, run_gpu
from workloads import Case, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _spec(seed=0):
    return dict(B=3, Hq=16, Hkv=4, D=128, P=16, lens=("fixed", 1), seed=seed)


def _healthy_call_still_works():
    case = make_case(_spec(8), seq_lens=[40, 700, 3])
    out, lse = run_gpu(case)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL


@pytest.mark.parametrize("bad_id", [-1, 1 << 30, "num_pages"])
def test_bad_page_index_is_reported_not_faulted(bad_id):
    case = make_case(_spec(1), seq_lens=[100, 200, 50])
    bad = case.num_pages if bad_id == "num_pages" else bad_id
    case.block_table[1, 3] = bad
    out, lse = run_gpu(case, expect_status=-6)
    # the other sequences are unaffected
    eo, el = compare_with_oracle(case, out, lse, select=[(0, h) for h in range(16)] + [(2, h) for h in range(16)])
    assert eo <= OUT_TOL and el <= LSE_TOL
    _healthy_call_still_works()


def test_bad_seq_len_is_reported():
    case = make_case(_spec(2), seq_lens=[100, 200, 50])
    for bad in (case.max_pages * case.P + 5, -3):
        case.seq_lens[2] = bad
        out, lse = run_gpu(case, expect_status=-8)
        # an invalid length makes that sequence empty; the others are unaffected
        assert out[2].float().abs().max().item() == 0 and torch.isneginf(lse[2]).all()
        ref = Case(**case.__dict__)
        ref.seq_lens = case.seq_lens.clone()
        ref.seq_lens[2] = 0
        eo, el = compare_with_oracle(ref, out, lse, select=[(0, h) for h in range(16)] + [(1, h) for h in range(16)])
        assert eo <= OUT_TOL and el <= LSE_TOL
    _healthy_call_still_works()


def test_bounded_wait_times_out_with_a_status():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pkv.pkv_selftest_wait_timeout(ws, timeout_us=2000)
    assert pkv.pkv_check_status(ws) == -7
    pkv.pkv_reset_status(ws)
    assert pkv.pkv_check_status(ws) == 0
    _healthy_call_still_works()


def test_workspace_too_small_is_rejected_before_launch():
    case = make_case(_spec(3), seq_lens=[5000, 10, 10]).to("cuda")
    need = pkv.paged_decode_attn_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages)
    assert need > 256
    ws = torch.zeros(need - 16, dtype=torch.uint8, device="cuda")
    out = torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale,
                              out, None, ws)
    assert e.value.status == -4


def test_longest_first_order_with_ties_and_bad_lengths():
    # A grid of several waves (40 sequences x 8 kv heads x 12 splits on one GPU) runs its
    # sequences longest first, ranked on the device from seq_lens; equal lengths, empty
    # sequences and invalid lengths (ranked as empty, reported) keep every row where it belongs.
    lens = [700, 33, 700, 0, 1, 2500, 700, 64, 1000, 33] * 4
    case = make_case(dict(B=40, Hq=16, Hkv=8, D=64, P=16, lens=("fixed", 1), seed=21), seq_lens=lens, poison=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, num_splits=12)
    assert plan["grid_blocks"] > sms * plan["blocks_per_sm"]  # several waves: the longest-first order applies
    out, lse = run_gpu(case, num_splits=12)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    bad = Case(**case.__dict__)
    bad.seq_lens = case.seq_lens.clone()
    bad.seq_lens[7] = -5
    bad.seq_lens[12] = case.max_pages * case.P + 1
    out, lse = run_gpu(bad, num_splits=12, expect_status=-8)
    ref = Case(**case.__dict__)
    ref.seq_lens = case.seq_lens.clone()
    ref.seq_lens[7] = 0
    ref.seq_lens[12] = 0
    eo, el = compare_with_oracle(ref, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
