"""Parity of the CUDA path (through the C-ABI) with the CPU fp64 oracle.

Bars: max |out - oracle| <= 1.5e-2 on bf16 outputs, max |lse - oracle| <= 1e-3
on f32 LSE, and results at different split counts within 2e-3 of each other.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import (LSE_TOL, OUT_TOL, SPLIT_TOL, compare_with_oracle, decode_oracle_rows, max_abs_diff, run_gpu,
                      sample_rows, split_straddle_check)
from workloads import CONFIG_ORDER, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _spec(B, Hq, Hkv, D, P, seed=0, **kw):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed, **kw)


# Small cases the oracle checks in full: several stages and splits, ragged tails,
# every head dim, group sizes 1..32, page sizes 8..256, NaN in every unused slot.
SMALL = [
    # B, Hq, Hkv, D, P, lens
    (1, 8, 2, 64, 16, [256]),
    (3, 8, 2, 64, 8, [1, 7, 8]),
    (4, 8, 8, 64, 16, [9, 15, 16, 17]),
    (3, 32, 8, 128, 16, [1, 300, 1000]),
    (5, 32, 8, 128, 16, [0, 17, 15, 16, 2500]),
    (2, 64, 8, 128, 16, [4097, 333]),
    (2, 16, 4, 128, 64, [63, 200]),
    (2, 16, 1, 128, 32, [130, 64]),
    (2, 32, 2, 256, 64, [2048, 77]),
    (3, 16, 2, 256, 16, [1, 500, 129]),
    (2, 64, 2, 128, 16, [700, 45]),
    (2, 32, 16, 64, 256, [600, 255]),
    (1, 4, 1, 256, 8, [1000]),
    (2, 24, 8, 128, 16, [100, 33]),   # G = 3 (padded head tile)
    (300, 8, 2, 128, 16, [(7 * i) % 97 for i in range(300)]),  # more sequences than the longest-first order ranks (128)
]


@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", SMALL, ids=lambda x: str(x).replace(" ", ""))
def test_small_cases_full_oracle(B, Hq, Hkv, D, P, lens):
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B * 7 + D), seq_lens=lens, poison=True)
    out, lse = run_gpu(case)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_workloads_sampled_oracle(name):
    """Every workload at full size, in the launch configuration the benchmark times."""
    case = make_case(name, device="cuda")
    out, lse = run_gpu(case)
    rows = sample_rows(case, n=24, seed=1) if name != "tiny" else None
    eo, el = compare_with_oracle(case, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (name, eo, el)
    # properties that hold at every row: finite, and a convex combination of V rows
    o = out.float()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert o.abs().max().item() <= case.v_cache.float().abs().max().item() * (1 + 2 ** -7)
    del case, out, lse
    torch.cuda.empty_cache()


def _split_counts_agree(case, counts, sample_n=12):
    """Runs the case at each split count (0 = the plan's own), then holds every pair to the
    split-count bar (f32 lse within 2e-3; bf16 out within 2e-3 except proven rounding straddles;
    mean |difference| within 2e-4) and each count's sampled rows to the oracle bars."""
    outs = [run_gpu(case, num_splits=s) for s in counts]
    host = [(o.float().cpu().numpy(), l.cpu().numpy()) for o, l in outs]
    del outs
    oracle_rows = decode_oracle_rows(case)
    for i in range(len(host)):
        for j in range(i + 1, len(host)):
            dl = max_abs_diff(host[i][1], host[j][1])
            assert dl <= SPLIT_TOL, (counts[i], counts[j], dl)  # f32 LSE: only the order of f32 sums differs
            n_big, d, mid = split_straddle_check(host[i][0], host[j][0], oracle_rows)
            mean_d = float(np.mean(np.abs(host[i][0] - host[j][0])))
            assert mean_d <= 2e-4, (counts[i], counts[j], mean_d, n_big, d)
    rows = sample_rows(case, sample_n)
    ref_o, ref_l = oracle_rows_with_lse(case, rows)
    idx = np.asarray(rows)
    for (o, l), s in zip(host, counts):
        eo = max_abs_diff(o[idx[:, 0], idx[:, 1]], ref_o)
        el = max_abs_diff(l[idx[:, 0], idx[:, 1]], ref_l)
        assert eo <= OUT_TOL and el <= LSE_TOL, (s, eo, el)


def oracle_rows_with_lse(case, rows):
    q, k, v, bt, sl = case.host_bits()
    return oracle.paged_decode(q, k, v, bt, sl, case.scale, select=rows)


@pytest.mark.parametrize("case_args", [
    ("batch", None),
    (_spec(3, 32, 8, 128, 16, seed=3), [1, 1000, 5000]),
    (_spec(2, 32, 2, 256, 64, seed=4), [3000, 65]),
])
def test_split_count_invariance(case_args):
    spec, lens = case_args
    case = make_case(spec, seq_lens=lens, device="cuda") if lens else make_case(spec, device="cuda")
    max_tokens = case.max_pages * case.P
    _split_counts_agree(case, [1, 2, 0, max(3, max_tokens // 16)])


@pytest.mark.parametrize("name,counts", [("long", [0, 1, 2, 8]), ("ragged", [0, 1, 2])])
def test_split_count_invariance_full_size(name, counts):
    """The full long-context and ragged workloads at the plan's own split count (42 and 8 on a
    152-SM GB300; the long one merged in six batches) against one, two (and eight) splits:
    where the split count matters most."""
    case = make_case(name, device="cuda")
    plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages,
                          torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["num_splits"] > max(c for c in counts), plan["num_splits"]
    _split_counts_agree(case, counts, sample_n=16)
    del case
    torch.cuda.empty_cache()


def test_reruns_are_bitwise_identical():
    case = make_case("batch", device="cuda")
    a = run_gpu(case)
    b = run_gpu(case)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_physical_page_placement_does_not_matter():
    case = make_case(_spec(4, 32, 8, 128, 16, seed=9), seq_lens=[1000, 17, 333, 2049])
    out_a, lse_a = run_gpu(case, num_splits=3)
    rng = np.random.default_rng(3)
    new_pool = case.num_pages + 40
    perm = torch.from_numpy(rng.permutation(new_pool)[: case.num_pages].astype(np.int64))
    k2 = torch.full((new_pool,) + tuple(case.k_cache.shape[1:]), float("nan"), dtype=torch.bfloat16)
    v2 = k2.clone()
    k2[perm] = case.k_cache
    v2[perm] = case.v_cache
    bt = case.block_table.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], torch.full_like(bt, -1)).int()
    moved = make_case(_spec(4, 32, 8, 128, 16, seed=9), seq_lens=[1000, 17, 333, 2049])
    moved.k_cache, moved.v_cache, moved.block_table, moved.num_pages = k2, v2, bt2, new_pool
    out_b, lse_b = run_gpu(moved, num_splits=3)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16)) and torch.equal(lse_a, lse_b)


def test_lse_may_be_null():
    case = make_case(_spec(2, 8, 2, 64, 16, seed=1), seq_lens=[100, 3000])
    out_a, _ = run_gpu(case, with_lse=False)
    out_b, _ = run_gpu(case)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_single_token_returns_v_row_exactly():
    """With one key the softmax weight is exactly 1: out is that V row, bit for bit."""
    case = make_case(_spec(3, 16, 2, 128, 16, seed=5), seq_lens=[1, 1, 1], poison=True)
    out, lse = run_gpu(case)
    bt = case.block_table
    for b in range(3):
        for h in range(16):
            assert torch.equal(out[b, h].cpu().view(torch.int16), case.v_cache[bt[b, 0], 0, h // 8].view(torch.int16))


def test_graph_capture_replay():
    case = make_case(_spec(4, 32, 8, 128, 16, seed=2), seq_lens=[500, 4000, 17, 1200]).to("cuda")
    ws_bytes = pkv.paged_decode_attn_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
    args = (case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale, out, lse, ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.paged_decode_attn(*args)  # warm-up outside capture (tensor maps, attributes)
    torch.cuda.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_decode_attn(*args, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert pkv.pkv_check_status(ws) == 0


def test_split_kv_merge_matches_oracle():
    rng = np.random.default_rng(0)
    S, B, Hq = 5, 3, 8
    for D in (64, 128, 256):
        po = rng.standard_normal((S, B, Hq, D)).astype(np.float32)
        pl = (rng.standard_normal((S, B, Hq)) * 4).astype(np.float32)
        pl[1, 0, :] = -np.inf          # an empty split
        pl[:, 2, 3] = -np.inf          # a row whose splits are all empty
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        pkv.split_kv_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out, lse)
        torch.cuda.synchronize()
        ro, rl = oracle.merge(po.reshape(S, B * Hq, D).astype(np.float64), pl.reshape(S, B * Hq).astype(np.float64))
        assert max_abs_diff(out.float().cpu().numpy().reshape(B * Hq, D), ro) <= 1e-2
        assert max_abs_diff(lse.cpu().numpy().reshape(-1), rl) <= 1e-5
        assert np.isneginf(lse[2, 3].item()) and out[2, 3].abs().max().item() == 0


@pytest.mark.parametrize("case_args,splits", [
    (("batch", None), 0),
    ((_spec(3, 32, 8, 128, 16, seed=3), [1, 1000, 5000]), 2),
    ((_spec(3, 32, 8, 128, 16, seed=3), [1, 1000, 5000]), 3),
    ((_spec(3, 32, 8, 128, 16, seed=3), [1, 1000, 5000]), 8),
    ((_spec(2, 32, 2, 256, 64, seed=4), [3000, 65]), 4),
    ((_spec(3, 8, 2, 64, 16, seed=6), [700, 0, 33]), 5),
    ((_spec(2, 32, 2, 128, 16, seed=7), [2000, 900]), 6),
])
def test_cluster_merge_equals_workspace_merge(case_args, splits):
    """Splits merged inside a thread-block cluster (split 0's shared memory) give the same bits
    as the workspace merge: the same partials, combined by the same batched combine in split order."""
    spec, lens = case_args
    case = make_case(spec, seq_lens=lens, device="cuda") if lens else make_case(spec, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    prev = pkv.set_cluster_merge(True)
    try:
        plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, num_splits=splits)
        assert plan["merge_needed"] == 2, plan
        a_out, a_lse = run_gpu(case, num_splits=splits)
        pkv.set_cluster_merge(False)
        plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, num_splits=splits)
        assert plan["merge_needed"] == 1, plan
        b_out, b_lse = run_gpu(case, num_splits=splits)
    finally:
        pkv.set_cluster_merge(prev)
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse.view(torch.int32), b_lse.view(torch.int32))
    eo, el = compare_with_oracle(case, a_out, a_lse, select=sample_rows(case, 12))
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("adaptive", [True, False])
@pytest.mark.parametrize("lens", [[2048, 1500, 3000, 77], [1, 0, 40000, 9], [3000, 40, 2000, 70000]])
def test_adaptive_split_count_on_a_wide_table(lens, adaptive):
    """A block table far wider than the batch's sequences (a pool sized for long contexts): the plan
    sizes its splits for the full width; with the adaptive split count the kernel re-sizes them
    from the actual lengths (more, shorter splits).  Against the oracle in full, and against one
    split (the straddle check)."""
    case = make_case(_spec(4, 64, 8, 128, 16, seed=61, max_pages=8192), seq_lens=lens, poison=True, device="cuda")
    plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages,
                          torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["num_splits"] > 1 and plan["chunk_tokens"] > 2048, plan
    prev = pkv.set_adaptive_splits(adaptive)
    try:
        out, lse = run_gpu(case)
        out2, _ = run_gpu(case)  # the merge counters return to 0
    finally:
        pkv.set_adaptive_splits(prev)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    one_o, one_l = run_gpu(case, num_splits=1)
    split_straddle_check(out.float().cpu().numpy(), one_o.float().cpu().numpy(), decode_oracle_rows(case))
    assert max_abs_diff(lse.cpu().numpy(), one_l.cpu().numpy()) <= SPLIT_TOL


@pytest.mark.parametrize("name", ["batch", "ragged", "long"])
def test_workloads_with_adaptive_splits(name):
    """The full-size workloads with the adaptive split count switched on: sampled rows against the
    oracle, and the whole output held to the split-count bar against the planned split (the two
    calls differ at most in where the splits end, which only reorders the f32 sums)."""
    case = make_case(name, device="cuda")
    base_o, base_l = run_gpu(case)
    prev = pkv.set_adaptive_splits(True)
    try:
        out, lse = run_gpu(case)
    finally:
        pkv.set_adaptive_splits(prev)
    eo, el = compare_with_oracle(case, out, lse, select=sample_rows(case, n=16, seed=5))
    assert eo <= OUT_TOL and el <= LSE_TOL, (name, eo, el)
    assert max_abs_diff(lse.cpu().numpy(), base_l.cpu().numpy()) <= SPLIT_TOL
    split_straddle_check(out.float().cpu().numpy(), base_o.float().cpu().numpy(), decode_oracle_rows(case))
    del case, out, lse, base_o, base_l
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", SMALL, ids=lambda x: str(x).replace(" ", ""))
def test_small_cases_with_adaptive_splits(B, Hq, Hkv, D, P, lens):
    """The small cases again with the adaptive split count switched on (tables wider than the
    longest sequence where the shape allows), against the oracle in full."""
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B * 7 + D, max_pages=max(1, 2 * max(lens) // P + 3)),
                     seq_lens=lens, poison=True)
    prev = pkv.set_adaptive_splits(True)
    try:
        out, lse = run_gpu(case)
    finally:
        pkv.set_adaptive_splits(prev)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
