"""Several query rows per sequence (multi-token decode, chunked paged prefill) on the GPU,
through the C-ABI, against the CPU oracle.

Bars: max |out - oracle| <= 1.5e-2, max |lse - oracle| <= 1e-3; one row per request
reproduces the decode kernel bit for bit; split counts agree to the split-count bar.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, max_abs_diff, run_gpu, split_invariance_violation, split_straddle_check
from workloads import Case, make_prefill_case, used_slot_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _spec(B, Hq, Hkv, D, P, seed=0):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed)


def run_prefill(case, causal=True, num_splits=0, fp8=None, expect_status=0, max_q_len=None):
    c = case if case.q.is_cuda else case.to("cuda")
    q_lens = np.diff(case.qo_indptr.cpu().numpy())
    mq = int(max_q_len if max_q_len is not None else max(1, q_lens.max() if q_lens.size else 1))
    total_q = c.q.shape[0]
    cache = "fp8" if fp8 is not None else "bf16"
    ws = torch.zeros(pkv.paged_prefill_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, total_q, mq,
                                                           num_splits=num_splits, cache=cache),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((total_q, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((total_q, c.Hq), float("nan"), dtype=torch.float32, device="cuda")
    if fp8 is not None:
        k8, v8, ks, vs = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in fp8)
        pkv.paged_prefill_attn(c.q, k8, v8, c.qo_indptr, c.block_table, c.seq_lens, mq, c.scale, out, lse, ws,
                               causal=causal, num_splits=num_splits, fp8_scales=(ks, vs))
    else:
        pkv.paged_prefill_attn(c.q, c.k_cache, c.v_cache, c.qo_indptr, c.block_table, c.seq_lens, mq, c.scale, out,
                               lse, ws, causal=causal, num_splits=num_splits)
    status = pkv.pkv_check_status(ws)
    assert status == expect_status, "device status %s" % pkv.STATUS.get(status, status)
    return out, lse


def prefill_oracle_rows(case, causal=True):
    """oracle_rows for split_straddle_check on a several-rows case: (t, h) rows -> fp64 outputs."""
    q, k, v, bt, sl = case.host_bits()
    qo = case.qo_indptr.cpu().numpy()
    return lambda rows: oracle.paged_prefill(q, qo, bt, sl, case.scale, causal=causal, k_bits=k, v_bits=v,
                                             select=[tuple(r) for r in rows])[0]


def compare(case, out, lse, causal=True, fp8=None, select=None):
    q, k, v, bt, sl = case.host_bits()
    qo = case.qo_indptr.cpu().numpy()
    kw = dict(fp8=fp8) if fp8 is not None else dict(k_bits=k, v_bits=v)
    ro, rl = oracle.paged_prefill(q, qo, bt, sl, case.scale, causal=causal, select=select, **kw)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    if select is not None:
        idx = np.asarray(list(select))
        o, l = o[idx[:, 0], idx[:, 1]], l[idx[:, 0], idx[:, 1]]
    return max_abs_diff(o, ro), max_abs_diff(l, rl)


SMALL = [
    # B, Hq, Hkv, D, P, q_lens, kv_lens
    (2, 8, 2, 64, 16, [3, 5], [40, 300]),
    (3, 32, 8, 128, 16, [4, 1, 2], [1000, 17, 2]),      # 32 rows per group: one tile of 32
    (2, 32, 8, 128, 16, [7, 3], [64, 500]),            # 56 rows: two tiles
    (2, 16, 2, 128, 8, [1, 6], [9, 6]),               # a request as long as its cache
    (1, 8, 1, 256, 64, [12], [700]),
    (2, 16, 2, 256, 16, [2, 3], [129, 4000]),
    (3, 4, 4, 64, 32, [33, 1, 5], [60, 3, 5]),         # G = 1, 33 rows: two tiles
    (2, 8, 2, 128, 16, [6, 0], [2, 100]),              # 6 rows over 2 keys; an empty request
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", SMALL, ids=lambda x: str(x).replace(" ", ""))
def test_small_cases_full_oracle(B, Hq, Hkv, D, P, q_lens, kv_lens, causal):
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=B + D + sum(q_lens)), q_lens, kv_lens, poison=True)
    out, lse = run_prefill(case, causal=causal)
    eo, el = compare(case, out, lse, causal=causal)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", SMALL[:6], ids=lambda x: str(x).replace(" ", ""))
def test_fp8_cache(B, Hq, Hkv, D, P, q_lens, kv_lens):
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=7 * B + D), q_lens, kv_lens, poison=True)
    _, k, v, _, _ = case.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    unused = ~used_slot_mask(case)
    for sc in (ks, vs):
        sc.transpose(0, 2, 1)[unused] = np.nan
    out, lse = run_prefill(case, fp8=(k8, v8, ks, vs))
    eo, el = compare(case, out, lse, fp8=(k8, v8, ks, vs))
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("causal", [True, False])
def test_one_row_per_request_is_the_decode_kernel(causal):
    case = make_prefill_case(_spec(5, 32, 8, 128, 16, seed=3), [1] * 5, [1, 17, 300, 1024, 4000], poison=True)
    for splits in (0, 1, 3):
        o1, l1 = run_prefill(case, causal=causal, num_splits=splits)
        dcase = Case(**case.__dict__)
        o2, l2 = run_gpu(dcase, num_splits=splits)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_split_counts_agree():
    case = make_prefill_case(_spec(3, 32, 8, 128, 16, seed=4), [4, 2, 3], [3000, 1200, 64])
    ref = run_prefill(case, num_splits=1)
    rows = prefill_oracle_rows(case)
    for splits in (0, 3, 7, 20):  # 20: the in-kernel merge takes the splits in three batches
        out, lse = run_prefill(case, num_splits=splits)
        split_straddle_check(out.float().cpu().numpy(), ref[0].float().cpu().numpy(), rows)
        assert max_abs_diff(lse.cpu().numpy(), ref[1].cpu().numpy()) <= 2e-3


def test_malformed_row_ranges_are_skipped_and_reported():
    case = make_prefill_case(_spec(3, 8, 2, 64, 16, seed=5), [2, 3, 1], [50, 60, 70])
    good_o, good_l = run_prefill(case)
    bad = Case(**case.__dict__)
    bad.qo_indptr = torch.tensor([0, 2, 9, 6], dtype=torch.int32)  # request 1 claims rows 2..8 (past total_q = 6)
    out, lse = run_prefill(bad, expect_status=-9, max_q_len=3)
    # request 0 is untouched by the bad range; request 2's range (9 > 6 rows... negative length) is skipped too
    assert torch.equal(out[:2].view(torch.int16), good_o[:2].view(torch.int16))
    assert torch.isnan(out[2:].float()).all()  # never written


def test_multi_token_step_at_full_size():
    # the batch workload's shape with four new tokens per sequence (a speculative / multi-token step)
    case = make_prefill_case("batch", [4] * 8, None, device="cuda")
    out, lse = run_prefill(case)
    rows = [(t, h) for t in range(0, 32, 3) for h in (0, 13, 31)]
    eo, el = compare(case, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ------------------------------------------------------------------ the tensor-core path
# bf16 cache, D = 128, at least 128 (token, head) rows per (sequence, kv head) group

TC = [
    # B, Hq, Hkv, D, P, q_lens, kv_lens
    (3, 32, 8, 128, 16, [40, 33, 64], [40, 500, 2000]),   # G = 4: 160, 132, 256 rows
    (2, 8, 1, 128, 64, [20, 17], [300, 17]),               # G = 8, a request as long as its cache
    (1, 16, 2, 128, 8, [130], [130]),                      # 1040 rows: 9 tiles, 8-key pages
    (2, 32, 8, 128, 256, [64, 3], [600, 5]),               # 256-key pages; a short request in the batch
    (2, 16, 4, 128, 32, [70, 0], [70, 40]),                # an empty request
    (2, 16, 2, 128, 64, [40, 9], [3000, 9]),               # 320 rows: a 256-row CTA whose second tile is partial
    (1, 32, 8, 128, 16, [96], [96]),                       # 384 rows, causal from the first key
    (2, 64, 8, 128, 16, [8, 5], [3000, 40]),               # G = 8: 64 and 40 rows, one partial tile each
    (3, 32, 8, 128, 32, [9, 12, 1], [500, 12, 700]),       # G = 4: 36, 48 and 4 rows
    (1, 32, 4, 128, 16, [5], [9000]),                      # 40 rows over a 9000-key table (key splits)
]


@pytest.mark.parametrize("mode", ["always", "rows128"])  # 256 rows per CTA where the group has them; 128
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", TC, ids=lambda x: str(x).replace(" ", ""))
def test_tensor_core_path_full_oracle(B, Hq, Hkv, D, P, q_lens, kv_lens, causal, mode):
    pkv.set_prefill_tensor_cores(mode)
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=3 * B + P + sum(q_lens)), q_lens, kv_lens, poison=True)
    out, lse = run_prefill(case, causal=causal)
    eo, el = compare(case, out, lse, causal=causal)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("q_lens,kv_lens,table_keys,kernel", [
    ([8, 5], [3000, 40], 4096, "off"),        # 64 rows, a 4096-key table: the mma.sync kernel
    ([8, 5], [3000, 40], 8192, "rows128"),    # the same rows, an 8192-key table: the 128-row tensor-core kernel
    ([4, 2], [9000, 40], 9008, "off"),        # 32 rows fit one mma.sync block whatever the table
])
def test_auto_routing_of_short_groups(q_lens, kv_lens, table_keys, kernel):
    # auto takes the tensor cores for groups of 33-127 rows only on tables of 8192 keys or more: its
    # result equals, bit for bit, the one of the kernel the rule names, and matches the oracle
    case = make_prefill_case(dict(_spec(2, 64, 8, 128, 16, seed=41), max_pages=table_keys // 16), q_lens, kv_lens,
                             poison=True)
    assert case.max_pages * case.P == table_keys
    pkv.set_prefill_tensor_cores("auto")
    out, lse = run_prefill(case)
    pkv.set_prefill_tensor_cores(kernel)
    ref_o, ref_l = run_prefill(case)
    assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)
    eo, el = compare(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def _fp8_pools(case):
    """Oracle-quantised pools of a case (NaN scales in every unused slot) and the bf16 case
    holding their dequantised values (exact: power-of-two scales)."""
    _, k, v, _, _ = case.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    unused = ~used_slot_mask(case)
    for sc in (ks, vs):
        sc.transpose(0, 2, 1)[unused] = np.nan
    deq = Case(**case.__dict__)
    for name, codes, sc in (("k_cache", k8, ks), ("v_cache", v8, vs)):
        vals = torch.from_numpy(oracle.dequantize_pool(codes, sc).astype(np.float32))
        setattr(deq, name, vals.to(torch.bfloat16).to(case.k_cache.device))
    return (k8, v8, ks, vs), deq


TC8 = TC  # page sizes 8-256, groups of 36-1040 rows, an empty request, key splits


@pytest.mark.parametrize("mode", ["rows128", "always", "auto"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", TC8, ids=lambda x: str(x).replace(" ", ""))
def test_fp8_tensor_core_path(B, Hq, Hkv, D, P, q_lens, kv_lens, causal, mode):
    # the fp8 cache on the 128-row tensor-core kernel: bit for bit the bf16 128-row kernel on the
    # dequantised cache (the converters write exactly the tiles its copies land), and the fp8 oracle
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=5 * B + P + sum(q_lens)), q_lens, kv_lens, poison=True)
    pools, deq = _fp8_pools(case)
    pkv.set_prefill_tensor_cores(mode)
    out, lse = run_prefill(case, causal=causal, fp8=pools)
    eo, el = compare(case, out, lse, causal=causal, fp8=pools)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    rows = max(q_lens) * (Hq // Hkv)
    if mode != "auto" or rows >= 128 or case.max_pages * P >= 8192:  # the call took the tensor cores
        pkv.set_prefill_tensor_cores("rows128")
        ref_o, ref_l = run_prefill(deq, causal=causal)
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)


def test_fp8_tensor_core_bad_page_and_key_splits():
    case = make_prefill_case(_spec(2, 16, 2, 128, 16, seed=23), [40, 20], [9000, 300], poison=True)
    pools, deq = _fp8_pools(case)
    pkv.set_prefill_tensor_cores("rows128")
    for splits in (0, 3, 16):
        out, lse = run_prefill(case, num_splits=splits, fp8=pools)
        rows = [(t, h) for t in range(0, 60, 7) for h in (0, 5, 15)]
        eo, el = compare(case, out, lse, fp8=pools, select=rows)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)
        ref_o, ref_l = run_prefill(deq, num_splits=splits)
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)
    bad = Case(**case.__dict__)
    bt = case.block_table.clone()
    bt[1, 3] = case.num_pages + 7
    bad.block_table = bt
    out, lse = run_prefill(bad, fp8=pools, expect_status=-6)
    o0, _ = run_prefill(case, fp8=pools)
    assert torch.equal(out[:40].view(torch.int16), o0[:40].view(torch.int16))  # request 0 untouched
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mode", ["always", "rows128"])
def test_tensor_core_and_mma_sync_paths_agree(mode):
    case = make_prefill_case(_spec(2, 32, 8, 128, 16, seed=9), [80, 40], [1000, 300])
    pkv.set_prefill_tensor_cores("off")
    ref_o, ref_l = run_prefill(case)
    pkv.set_prefill_tensor_cores(mode)
    out, lse = run_prefill(case)
    excess, _, _ = split_invariance_violation(out.float().cpu().numpy(), ref_o.float().cpu().numpy(), tol=OUT_TOL)
    assert excess <= 0
    assert max_abs_diff(lse.cpu().numpy(), ref_l.cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("mode", ["always", "rows128"])
def test_tensor_core_path_bad_page_is_skipped_and_reported(mode):
    case = make_prefill_case(_spec(2, 32, 8, 128, 16, seed=10), [70, 40], [200, 300])
    bt = case.block_table.clone()
    bt[1, 3] = case.num_pages + 7
    bad = Case(**case.__dict__)
    bad.block_table = bt
    pkv.set_prefill_tensor_cores(mode)
    out, lse = run_prefill(bad, expect_status=-6)
    # request 0 is untouched; request 1 attends to its other keys only
    o0, l0 = run_prefill(case)
    assert torch.equal(out[:70].view(torch.int16), o0[:70].view(torch.int16))
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mode", ["always", "rows128"])
@pytest.mark.parametrize("splits", [0, 3, 16])
def test_tensor_core_key_splits(mode, splits):
    # 9000 keys: several 32-tile chunks per group, merged by the last split; a short request beside it
    case = make_prefill_case(_spec(2, 16, 2, 128, 16, seed=21), [40, 20], [9000, 300], poison=True)
    pkv.set_prefill_tensor_cores(mode)
    out, lse = run_prefill(case, num_splits=splits)
    rows = [(t, h) for t in range(0, 60, 7) for h in (0, 5, 15)]
    eo, el = compare(case, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("mode", ["always", "rows128"])
def test_tensor_core_splits_reuse_the_workspace(mode):
    # the merge counters wrap to 0 after each call: repeated calls on one workspace agree bit for bit
    c = make_prefill_case(_spec(2, 16, 2, 128, 16, seed=22), [40, 33], [6000, 4500]).to("cuda")
    pkv.set_prefill_tensor_cores(mode)
    total_q, mq = c.q.shape[0], 40
    ws = torch.zeros(pkv.paged_prefill_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, total_q, mq,
                                                           num_splits=4), dtype=torch.uint8, device="cuda")
    results = []
    for _ in range(3):
        out = torch.full((total_q, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((total_q, c.Hq), float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_prefill_attn(c.q, c.k_cache, c.v_cache, c.qo_indptr, c.block_table, c.seq_lens, mq, c.scale, out,
                               lse, ws, num_splits=4)
        assert pkv.pkv_check_status(ws) == 0
        results.append((out, lse))
    for out, lse in results[1:]:
        assert torch.equal(out.view(torch.int16), results[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), results[0][1].view(torch.int32))
    ref = run_prefill(c, num_splits=1)
    split_straddle_check(results[0][0].float().cpu().numpy(), ref[0].float().cpu().numpy(), prefill_oracle_rows(c))
    assert max_abs_diff(results[0][1].cpu().numpy(), ref[1].cpu().numpy()) <= 2e-3


@pytest.mark.parametrize("workload,q_len", [("batch", 512), ("ragged", 64), ("long", 32)])
def test_tensor_core_path_at_full_size(workload, q_len):
    # the workloads and the routing bench.py times (auto: 256 rows per CTA, key splits on ragged and
    # long), sampled rows against the oracle, and a second call equal bit for bit
    from workloads import CONFIGS, draw_seq_lens
    spec = CONFIGS[workload]
    kv = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
    case = make_prefill_case(workload, [q_len] * spec["B"], kv, device="cuda")
    pkv.set_prefill_tensor_cores("auto")
    out, lse = run_prefill(case)
    out2, lse2 = run_prefill(case)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    total_q = case.q.shape[0]
    rows = [(t, h) for t in range(0, total_q, max(1, total_q // 16)) for h in (0, case.Hq // 2 + 1, case.Hq - 1)]
    rows += [(total_q - 1, 3)]  # the last token of the last request
    eo, el = compare(case, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("workload,q_len", [("batch", 512), ("ragged", 16), ("long", 8)])
def test_fp8_tensor_core_path_at_full_size(workload, q_len):
    # the fp8 cache on the tensor cores at the sizes and in the routing bench.py times (auto: the
    # 128-row kernel's fp8 instantiation; key splits on long), pools quantised by the oracle:
    # sampled rows against the fp8 oracle, and a second call equal bit for bit
    from workloads import CONFIGS, draw_seq_lens
    spec = CONFIGS[workload]
    kv = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
    case = make_prefill_case(workload, [q_len] * spec["B"], kv)
    _, k, v, _, _ = case.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    del k, v
    pools = (k8, v8, ks, vs)
    dcase = case.to("cuda")
    pkv.set_prefill_tensor_cores("auto")
    out, lse = run_prefill(dcase, fp8=pools)
    out2, lse2 = run_prefill(dcase, fp8=pools)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    total_q = case.q.shape[0]
    rows = [(t, h) for t in range(0, total_q, max(1, total_q // 12)) for h in (0, case.Hq // 2 + 1, case.Hq - 1)]
    rows += [(total_q - 1, 3)]
    eo, el = compare(case, out, lse, fp8=pools, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    del case, dcase, pools, out, lse, out2, lse2
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ the tensor-core path at D = 256
# bf16 cache: 128 rows per CTA, 64-key tiles (prefill_tc256_kernel)

TC256 = [
    # B, Hq, Hkv, D, P, q_lens, kv_lens
    (2, 32, 2, 256, 64, [8, 5], [2048, 300]),    # G = 16: 128 and 80 rows, 64-key pages (the big-page shape)
    (2, 16, 4, 256, 16, [40, 33], [500, 33]),    # G = 4: 160 and 132 rows, a request as long as its cache
    (1, 8, 1, 256, 8, [130], [130]),             # 1040 rows: 9 tiles, 8-key pages (two boxes per 16-key step)
    (2, 16, 2, 256, 128, [20, 0], [700, 9]),     # 128-key pages (64-key boxes), an empty request
    (2, 32, 4, 256, 32, [17, 16], [40, 16]),     # 136 and 128 rows over fewer than 64 keys: one partial tile
    (1, 16, 2, 256, 16, [9], [9000]),            # 72 rows over a 9000-key table: key splits
]


@pytest.mark.parametrize("mode", ["always", "auto"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", TC256, ids=lambda x: str(x).replace(" ", ""))
def test_tensor_core_path_d256_full_oracle(B, Hq, Hkv, D, P, q_lens, kv_lens, causal, mode):
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=7 * B + P + sum(q_lens)), q_lens, kv_lens, poison=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    try:
        pkv.set_prefill_tensor_cores(mode)
        rows = max(q_lens) * (Hq // Hkv)
        plan = pkv.prefill_plan_query(B, Hq, Hkv, D, P, case.max_pages, case.q.shape[0], max(q_lens), sms)
        takes_tc = rows > 32 and (mode == "always" or rows >= 128 or case.max_pages * P >= 8192)
        assert (plan["rows_per_block"] == 128 and plan["stage_tokens"] == 64) == takes_tc, plan
        out, lse = run_prefill(case, causal=causal)
    finally:
        pkv.set_prefill_tensor_cores("auto")
    eo, el = compare(case, out, lse, causal=causal)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_d256_tensor_core_and_mma_sync_paths_agree():
    case = make_prefill_case(_spec(2, 32, 2, 256, 64, seed=51), [8, 6], [1500, 400])
    try:
        pkv.set_prefill_tensor_cores("off")
        ref_o, ref_l = run_prefill(case)
        pkv.set_prefill_tensor_cores("always")
        out, lse = run_prefill(case)
    finally:
        pkv.set_prefill_tensor_cores("auto")
    excess, _, _ = split_invariance_violation(out.float().cpu().numpy(), ref_o.float().cpu().numpy(), tol=OUT_TOL)
    assert excess <= 0
    assert max_abs_diff(lse.cpu().numpy(), ref_l.cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("splits", [0, 3, 16])
def test_d256_tensor_core_key_splits_and_bad_page(splits):
    case = make_prefill_case(_spec(2, 32, 2, 256, 16, seed=52), [8, 4], [9000, 300], poison=True)
    try:
        pkv.set_prefill_tensor_cores("always")
        out, lse = run_prefill(case, num_splits=splits)
        rows = [(t, h) for t in range(12) for h in (0, 7, 31)]
        eo, el = compare(case, out, lse, select=rows)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)
        out2, lse2 = run_prefill(case, num_splits=splits)  # the merge counters return to 0
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        bad = Case(**case.__dict__)
        bt = case.block_table.clone()
        bt[1, 2] = case.num_pages + 3
        bad.block_table = bt
        o_bad, _ = run_prefill(bad, num_splits=splits, expect_status=-6)
        assert torch.equal(o_bad[:8].view(torch.int16), out[:8].view(torch.int16))  # request 0 untouched
        assert torch.isfinite(o_bad.float()).all()
    finally:
        pkv.set_prefill_tensor_cores("auto")


def test_d256_tensor_core_path_at_full_size():
    # the big-page G = 16 workload with 8 new tokens per sequence (128 rows per group): auto takes the
    # D = 256 tensor-core kernel; sampled rows against the oracle, a second call equal bit for bit
    from workloads import CONFIGS, draw_seq_lens
    spec = CONFIGS["bigpage_g16"]
    kv = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
    case = make_prefill_case("bigpage_g16", [8] * spec["B"], kv, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pkv.set_prefill_tensor_cores("auto")
    plan = pkv.prefill_plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, case.q.shape[0], 8, sms)
    assert plan["rows_per_block"] == 128 and plan["stage_tokens"] == 64, plan
    out, lse = run_prefill(case)
    out2, lse2 = run_prefill(case)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    total_q = case.q.shape[0]
    rows = [(t, h) for t in range(0, total_q, max(1, total_q // 16)) for h in (0, 17, case.Hq - 1)]
    rows += [(total_q - 1, 5)]
    eo, el = compare(case, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# fp8 cache at D = 256: the same kernel's instantiation with converter warps (codes and scales
# staged by TMA, dequantised to bf16 tiles in the layout the bf16 copies land)

@pytest.mark.parametrize("mode", ["always", "auto"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_lens,kv_lens", TC256, ids=lambda x: str(x).replace(" ", ""))
def test_fp8_tensor_core_path_d256(B, Hq, Hkv, D, P, q_lens, kv_lens, causal, mode):
    # against the fp8 oracle, and bit for bit the bf16 kernel on the dequantised cache where the
    # call took the tensor cores (the converters write exactly the tiles its copies land)
    case = make_prefill_case(_spec(B, Hq, Hkv, D, P, seed=9 * B + P + sum(q_lens)), q_lens, kv_lens, poison=True)
    pools, deq = _fp8_pools(case)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    try:
        pkv.set_prefill_tensor_cores(mode)
        rows = max(q_lens) * (Hq // Hkv)
        plan = pkv.prefill_plan_query(B, Hq, Hkv, D, P, case.max_pages, case.q.shape[0], max(q_lens), sms, cache="fp8")
        takes_tc = rows > 32 and (mode == "always" or rows >= 128 or case.max_pages * P >= 8192)
        assert (plan["rows_per_block"] == 128 and plan["stage_tokens"] == 64) == takes_tc, plan
        out, lse = run_prefill(case, causal=causal, fp8=pools)
        eo, el = compare(case, out, lse, causal=causal, fp8=pools)
        assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
        if takes_tc:
            ref_o, ref_l = run_prefill(deq, causal=causal)
            assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)
    finally:
        pkv.set_prefill_tensor_cores("auto")


@pytest.mark.parametrize("splits", [0, 3, 16])
def test_fp8_d256_tensor_core_key_splits_and_bad_page(splits):
    case = make_prefill_case(_spec(2, 32, 2, 256, 16, seed=53), [8, 4], [9000, 300], poison=True)
    pools, deq = _fp8_pools(case)
    try:
        pkv.set_prefill_tensor_cores("always")
        out, lse = run_prefill(case, num_splits=splits, fp8=pools)
        rows = [(t, h) for t in range(12) for h in (0, 7, 31)]
        eo, el = compare(case, out, lse, fp8=pools, select=rows)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)
        ref_o, ref_l = run_prefill(deq, num_splits=splits)
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)
        out2, _ = run_prefill(case, num_splits=splits, fp8=pools)  # the merge counters return to 0
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        bad = Case(**case.__dict__)
        bt = case.block_table.clone()
        bt[1, 2] = case.num_pages + 3
        bad.block_table = bt
        o_bad, _ = run_prefill(bad, num_splits=splits, fp8=pools, expect_status=-6)
        assert torch.equal(o_bad[:8].view(torch.int16), out[:8].view(torch.int16))  # request 0 untouched
        assert torch.isfinite(o_bad.float()).all()
    finally:
        pkv.set_prefill_tensor_cores("auto")


def test_fp8_d256_tensor_core_path_at_full_size():
    # the big-page G = 16 workload on the fp8 cache with 8 new tokens per sequence (128 rows per
    # group): auto takes the D = 256 tensor-core kernel; sampled rows against the fp8 oracle, a
    # second call equal bit for bit
    from workloads import CONFIGS, draw_seq_lens
    spec = CONFIGS["bigpage_g16"]
    kv = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
    case = make_prefill_case("bigpage_g16", [8] * spec["B"], kv)
    _, k, v, _, _ = case.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    del k, v
    pools = (k8, v8, ks, vs)
    dcase = case.to("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pkv.set_prefill_tensor_cores("auto")
    plan = pkv.prefill_plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, case.q.shape[0], 8, sms,
                                  cache="fp8")
    assert plan["rows_per_block"] == 128 and plan["stage_tokens"] == 64 and plan["warps"] == 11, plan
    out, lse = run_prefill(dcase, fp8=pools)
    out2, lse2 = run_prefill(dcase, fp8=pools)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    total_q = case.q.shape[0]
    rows = [(t, h) for t in range(0, total_q, max(1, total_q // 16)) for h in (0, 17, case.Hq - 1)]
    rows += [(total_q - 1, 5)]
    eo, el = compare(case, out, lse, fp8=pools, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    del case, dcase, pools, out, lse, out2, lse2
    torch.cuda.empty_cache()
