"""The FP8 (e4m3) KV cache on the GPU, through the C-ABI, against the CPU oracle.

Three bars:
  - decode over an fp8 cache matches the oracle's fp8 decode (out <= 1.5e-2, lse <= 1e-3);
  - it agrees with the bf16 kernel run with the same split count on the dequantised
    cache: lse to 1e-5 (the scores are the same products, summed in another order),
    out to the output bar with a mean difference below 1e-3 (the bf16 kernel rounds
    the probabilities to bf16, 2^-9 relative, the fp8 kernel to f16, 2^-12);
  - the quantise-and-append write is byte work: codes and scales equal the oracle's bit
    for bit, everywhere in the pools.
The fp8 pools of the decode tests are quantised by the oracle, never by the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import (LSE_TOL, OUT_TOL, SPLIT_TOL, max_abs_diff, run_gpu, sample_rows, split_invariance_violation,
                      split_straddle_check)
from test_parity import SMALL
from workloads import CONFIG_ORDER, Case, bf16_bits, bits_to_bf16, make_case, used_slot_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _spec(B, Hq, Hkv, D, P, seed=0, **kw):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed, **kw)


class Fp8Pools:
    """Oracle-quantised fp8 pools of a bf16 case (host numpy)."""

    def __init__(self, case, poison_scales=True):
        _, k, v, _, _ = case.host_bits()
        self.k8, self.ks = oracle.quantize_pool(k)
        self.v8, self.vs = oracle.quantize_pool(v)
        if poison_scales:  # unused slots: NaN codes already (NaN rows), NaN scales too
            unused = ~used_slot_mask(case)
            for s in (self.ks, self.vs):
                s.transpose(0, 2, 1)[unused] = np.nan

    def device(self):
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        return t(self.k8), t(self.v8), t(self.ks), t(self.vs)

    def dequantised_case(self, case):
        """The bf16 case holding the dequantised values (exact: power-of-two scales)."""
        c = Case(**case.__dict__)
        for name, codes, sc in (("k_cache", self.k8, self.ks), ("v_cache", self.v8, self.vs)):
            vals = torch.from_numpy(oracle.dequantize_pool(codes, sc).astype(np.float32))
            b = vals.to(torch.bfloat16)
            fin = torch.isfinite(vals)
            assert torch.equal(b.float()[fin], vals[fin])  # exactly representable
            setattr(c, name, b.to(case.k_cache.device))
        return c


def run_fp8(case, pools, num_splits=0, with_lse=True, expect_status=0):
    c = case if case.q.is_cuda else case.to("cuda")
    k8, v8, ks, vs = pools.device()
    ws_bytes = pkv.paged_decode_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, num_splits=num_splits,
                                                    cache="fp8")
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    pkv.paged_decode_attn_fp8(c.q, k8, v8, ks, vs, c.block_table, c.seq_lens, c.scale, out, lse, ws,
                              num_splits=num_splits)
    status = pkv.pkv_check_status(ws)
    assert status == expect_status, "device status %s" % pkv.STATUS.get(status, status)
    return out, lse


def compare_fp8_with_oracle(case, pools, out, lse, select=None):
    q, _, _, bt, sl = case.host_bits()
    ref_o, ref_l = oracle.paged_decode_fp8(q, pools.k8, pools.v8, pools.ks, pools.vs, bt, sl, case.scale,
                                           select=select)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    if select is not None:
        idx = np.asarray(list(select))
        o, l = o[idx[:, 0], idx[:, 1]], l[idx[:, 0], idx[:, 1]]
    return max_abs_diff(o, ref_o), max_abs_diff(l, ref_l)


def assert_agrees_with_bf16(a_out, a_lse, b_out, b_lse):
    a, b = a_out.float().cpu().numpy(), b_out.float().cpu().numpy()
    excess, _, _ = split_invariance_violation(a, b, tol=OUT_TOL)  # OUT_TOL, or one bf16 step of the output
    assert excess <= 0, excess
    assert float(np.mean(np.abs(a - b))) <= 1e-3
    assert max_abs_diff(a_lse.cpu().numpy(), b_lse.cpu().numpy()) <= 1e-5


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", SMALL, ids=lambda x: str(x).replace(" ", ""))
def test_fp8_small_cases_full_oracle(B, Hq, Hkv, D, P, lens):
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B * 11 + D), seq_lens=lens, poison=True)
    pools = Fp8Pools(case)
    out, lse = run_fp8(case, pools)
    eo, el = compare_fp8_with_oracle(case, pools, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", SMALL[::2], ids=lambda x: str(x).replace(" ", ""))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fp8_agrees_with_bf16_on_dequantised_cache(B, Hq, Hkv, D, P, lens, splits):
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B * 13 + D), seq_lens=lens, poison=True)
    pools = Fp8Pools(case)
    o8, l8 = run_fp8(case, pools, num_splits=splits)
    ob, lb = run_gpu(pools.dequantised_case(case), num_splits=splits)
    assert_agrees_with_bf16(o8, l8, ob, lb)


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_fp8_workloads_sampled_oracle(name):
    """Every workload at full size with an fp8 cache, in the benchmark's launch configuration."""
    case = make_case(name)
    pools = Fp8Pools(case, poison_scales=False)
    dcase = case.to("cuda")
    out, lse = run_fp8(dcase, pools)
    rows = sample_rows(case, n=24, seed=2) if name != "tiny" else None
    eo, el = compare_fp8_with_oracle(case, pools, out, lse, select=rows)
    assert eo <= OUT_TOL and el <= LSE_TOL, (name, eo, el)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    if name in ("tiny", "batch", "ragged"):  # against the bf16 kernel where the host copies stay small
        ob, lb = run_gpu(pools.dequantised_case(case))
        assert_agrees_with_bf16(out, lse, ob, lb)
    del case, dcase, pools, out, lse
    torch.cuda.empty_cache()


def test_fp8_bad_page_ids_and_lengths():
    case = make_case(_spec(3, 16, 4, 128, 16, seed=21), seq_lens=[40, 70, 5])
    pools = Fp8Pools(case)
    bt = case.block_table.clone()
    bt[1, 2] = case.num_pages + 5  # a used page of sequence 1 is out of range
    bad = Case(**case.__dict__)
    bad.block_table = bt
    out, lse = run_fp8(bad, pools, expect_status=-6)
    # the page is skipped: sequence 1 attends to its other keys only
    lens = case.seq_lens.numpy()
    keep = np.ones(lens[1], bool)
    keep[32:48] = False
    q, _, _, _, _ = case.host_bits()
    k8 = pools.k8.copy()
    # the oracle reads the same keys when the skipped page's keys are moved past the length
    idx = np.flatnonzero(keep)
    pages = case.block_table.numpy()[1]
    phys = [(int(pages[j // 16]), j % 16) for j in idx]
    nk8 = np.zeros((len(idx), 1, 4, 128), np.uint8)
    nv8 = np.zeros_like(nk8)
    nks = np.zeros((len(idx), 4, 1), np.float32)
    nvs = np.zeros_like(nks)
    for i, (pg, sl) in enumerate(phys):
        nk8[i, 0], nv8[i, 0] = pools.k8[pg, sl], pools.v8[pg, sl]
        nks[i, :, 0], nvs[i, :, 0] = pools.ks[pg, :, sl], pools.vs[pg, :, sl]
    ro, rl = oracle.paged_decode_fp8(q[1:2], nk8, nv8, nks, nvs, np.arange(len(idx), dtype=np.int32)[None],
                                     np.array([len(idx)], np.int32), case.scale)
    assert max_abs_diff(out[1].float().cpu().numpy(), ro[0]) <= OUT_TOL
    assert max_abs_diff(lse[1].cpu().numpy(), rl[0]) <= LSE_TOL
    # a length past the table makes that sequence empty
    bad2 = Case(**case.__dict__)
    bad2.seq_lens = torch.tensor([40, 70, 10_000], dtype=torch.int32)
    out2, lse2 = run_fp8(bad2, pools, expect_status=-8)
    assert torch.all(out2[2].float().cpu() == 0) and torch.all(torch.isinf(lse2[2].cpu()))


def test_fp8_empty_and_single_token():
    case = make_case(_spec(3, 8, 2, 64, 16, seed=5), seq_lens=[0, 1, 16], poison=True)
    pools = Fp8Pools(case)
    out, lse = run_fp8(case, pools)
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    # one key: the output is that key's dequantised V row, rounded to bf16
    pg = int(case.block_table[1, 0])
    vrow = oracle.dequantize_pool(pools.v8, pools.vs)[pg, 0]  # [Hkv, D]
    want = torch.from_numpy(vrow.astype(np.float32)).to(torch.bfloat16).repeat_interleave(4, dim=0)
    assert torch.equal(out[1].cpu(), want)
    eo, el = compare_fp8_with_oracle(case, pools, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL


# ------------------------------------------------------------------ quantise-and-append

def _wide_rows(shape, seed):
    """bf16 rows spanning many magnitudes: per-row powers of two, zero rows, subnormal-code values."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    rows = x.view(-1, shape[-1])
    e = torch.randint(-30, 30, (rows.shape[0], 1), generator=g).float()
    rows.mul_(torch.exp2(e))
    rows[::17] = 0.0
    rows[5::23, : shape[-1] // 2] *= 2.0 ** -12  # values far below the row maximum: subnormal codes, zeros
    rows[7::29] *= 2.0 ** 60                        # past the largest scale: saturated codes
    rows[11::31] *= 2.0 ** -90                      # below the smallest scale
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("Hkv,D,P", [(2, 64, 8), (8, 128, 16), (2, 256, 64), (1, 128, 256)])
def test_quantize_pool_bit_exact(Hkv, D, P):
    num_pages = 37
    k = _wide_rows((num_pages, P, Hkv, D), seed=D + P)
    v = _wide_rows((num_pages, P, Hkv, D), seed=D + P + 1)
    k8, v8, ks, vs = pkv.quantize_pool_fp8(k.cuda(), v.cuda())
    torch.cuda.synchronize()
    for gpu_c, gpu_s, src in ((k8, ks, k), (v8, vs, v)):
        rc, rs = oracle.quantize_pool(bf16_bits(src))
        assert np.array_equal(gpu_c.cpu().numpy(), rc)
        assert np.array_equal(gpu_s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("B,Hkv,D,P", [(3, 2, 64, 8), (5, 8, 128, 16), (300, 1, 256, 64)])
def test_fp8_append_bit_exact(B, Hkv, D, P):
    num_pages, max_pages = B + 3, 3
    g = np.random.default_rng(B + D)
    k8 = g.integers(0, 256, (num_pages, P, Hkv, D), dtype=np.uint8)
    v8 = g.integers(0, 256, (num_pages, P, Hkv, D), dtype=np.uint8)
    ks = g.standard_normal((num_pages, Hkv, P)).astype(np.float32)
    vs = g.standard_normal((num_pages, Hkv, P)).astype(np.float32)
    bt = np.stack([g.permutation(num_pages)[:max_pages] for _ in range(B)]).astype(np.int32)
    pos = g.integers(0, max_pages * P, B).astype(np.int32)
    pos[:: 4] = -1  # nothing to append for these
    pos[0] = max_pages * P - 1
    kn = _wide_rows((B, Hkv, D), seed=3)
    vn = _wide_rows((B, Hkv, D), seed=4)
    # one writer per (page, slot): keep the first sequence that targets a cell
    seen = set()
    for b in range(B):
        if pos[b] < 0:
            continue
        cell = (int(bt[b, pos[b] // P]), int(pos[b] % P))
        if cell in seen:
            pos[b] = -1
        seen.add(cell)
    dev = [torch.from_numpy(a.copy()).cuda() for a in (k8, v8, ks, vs)]
    pkv.paged_kv_append_fp8(kn.cuda(), vn.cuda(), torch.from_numpy(bt).cuda(), torch.from_numpy(pos).cuda(), *dev)
    torch.cuda.synchronize()
    rk, rv, rks, rvs, rej = oracle.kv_append_fp8(bf16_bits(kn), bf16_bits(vn), bt, pos, k8, v8, ks, vs)
    assert rej == 0
    assert np.array_equal(dev[0].cpu().numpy(), rk) and np.array_equal(dev[1].cpu().numpy(), rv)
    assert np.array_equal(dev[2].cpu().numpy().view(np.uint32), rks.view(np.uint32))
    assert np.array_equal(dev[3].cpu().numpy().view(np.uint32), rvs.view(np.uint32))


def test_fp8_append_reports_bad_positions_and_pages():
    P, Hkv, D, num_pages = 16, 2, 128, 6
    k8 = np.zeros((num_pages, P, Hkv, D), np.uint8)
    ks = np.ones((num_pages, Hkv, P), np.float32)
    bt = np.array([[0, 1], [2, num_pages + 4], [3, 4]], np.int32)
    kn = _wide_rows((3, Hkv, D), seed=9)
    for pos, want in (([3, 5, 2 * P], -8), ([3, P + 1, 7], -6)):
        dev = [torch.from_numpy(a.copy()).cuda() for a in (k8, k8, ks, ks)]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.paged_kv_append_fp8(kn.cuda(), kn.cuda(), torch.from_numpy(bt).cuda(),
                                torch.tensor(pos, dtype=torch.int32).cuda(), *dev, status=status)
        assert int(status.item()) == want
        rk, _, rks, _, rej = oracle.kv_append_fp8(bf16_bits(kn), bf16_bits(kn), bt, np.array(pos, np.int32),
                                                  k8, k8, ks, ks)
        assert rej == 1
        assert np.array_equal(dev[0].cpu().numpy(), rk)
        assert np.array_equal(dev[2].cpu().numpy().view(np.uint32), rks.view(np.uint32))


def test_fp8_append_then_decode():
    # one serving step over an fp8 cache: quantise-and-append the new token, then decode L + 1 keys
    case = make_case(_spec(4, 32, 8, 128, 16, seed=31), seq_lens=[31, 32, 1000, 1])
    lens = case.seq_lens.numpy()
    bt = np.concatenate([case.block_table.numpy(), np.full((4, 1), -1, np.int32)], axis=1)
    extra = [b for b in range(4) if lens[b] % 16 == 0]
    for i, b in enumerate(extra):
        bt[b, lens[b] // 16] = case.num_pages + i
    case.k_cache = torch.cat([case.k_cache, torch.zeros((len(extra),) + tuple(case.k_cache.shape[1:]),
                                                        dtype=torch.bfloat16)])
    case.v_cache = torch.cat([case.v_cache, torch.zeros_like(case.k_cache[: len(extra)])])
    case.num_pages += len(extra)
    case.max_pages += 1
    case.block_table = torch.from_numpy(bt)
    pools = Fp8Pools(case, poison_scales=False)
    g = torch.Generator().manual_seed(12)
    kn = torch.randn(4, 8, 128, generator=g).to(torch.bfloat16)  # the workloads' N(0, 1) rows
    vn = torch.randn(4, 8, 128, generator=g).to(torch.bfloat16)
    dev = list(pools.device())
    pkv.paged_kv_append_fp8(kn.cuda(), vn.cuda(), case.block_table.cuda(), torch.from_numpy(lens).cuda(), *dev)
    k8, v8, ks, vs, rej = oracle.kv_append_fp8(bf16_bits(kn), bf16_bits(vn), bt, lens, pools.k8, pools.v8,
                                               pools.ks, pools.vs)
    assert rej == 0
    stepped = Case(**case.__dict__)
    stepped.seq_lens = torch.from_numpy((lens + 1).astype(np.int32))
    after = Fp8Pools.__new__(Fp8Pools)
    after.k8, after.v8 = dev[0].cpu().numpy(), dev[1].cpu().numpy()
    after.ks, after.vs = dev[2].cpu().numpy(), dev[3].cpu().numpy()
    assert np.array_equal(after.k8, k8) and np.array_equal(after.vs.view(np.uint32), vs.view(np.uint32))
    out, lse = run_fp8(stepped, after)
    eo, el = compare_fp8_with_oracle(stepped, after, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL


@pytest.mark.parametrize("lens,splits", [([1, 1000, 5000], 4), ([1, 1000, 5000], 3), ([4000, 17, 2500], 7)])
def test_fp8_cluster_merge_equals_workspace_merge(lens, splits):
    """The fp8 cache's splits merged inside a thread-block cluster give the workspace merge's bits."""
    case = make_case(_spec(3, 32, 8, 128, 16, seed=41), seq_lens=lens, poison=True)
    pools = Fp8Pools(case)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    prev = pkv.set_cluster_merge(True)
    try:
        plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, num_splits=splits,
                              cache="fp8")
        assert plan["merge_needed"] == 2, plan
        a = run_fp8(case, pools, num_splits=splits)
        pkv.set_cluster_merge(False)
        b = run_fp8(case, pools, num_splits=splits)
    finally:
        pkv.set_cluster_merge(prev)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    eo, el = compare_fp8_with_oracle(case, pools, *a)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_fp8_group_32_at_head_dim_256():
    """G = 32 at D = 256 on the fp8 cache: two 16-head query tiles per group, against the fp8 oracle."""
    case = make_case(_spec(2, 64, 2, 256, 16, seed=29), seq_lens=[1200, 40], poison=True)
    pools = Fp8Pools(case)
    for splits in (1, 0, 5):
        out, lse = run_fp8(case, pools, num_splits=splits)
        eo, el = compare_fp8_with_oracle(case, pools, out, lse)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)


@pytest.mark.parametrize("lens", [[2048, 1500, 3000, 77], [1, 0, 40000, 9], [3000, 40, 2000, 70000]])
def test_fp8_adaptive_split_count_on_a_wide_table(lens):
    """The fp8 cache under the adaptive split count, on a block table far wider than the batch's
    sequences: against the fp8 oracle in full, repeatable bit for bit (the merge counters return
    to zero), and held to the split-count bar against one split."""
    case = make_case(_spec(4, 64, 8, 128, 16, seed=67, max_pages=8192), seq_lens=lens, poison=True)
    pools = Fp8Pools(case)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pkv.plan_query(case.B, case.Hq, case.Hkv, case.D, case.P, case.max_pages, sms, cache="fp8")
    assert plan["num_splits"] > 1 and plan["chunk_tokens"] > 2048, plan
    prev = pkv.set_adaptive_splits(True)
    try:
        out, lse = run_fp8(case, pools)
        out2, lse2 = run_fp8(case, pools)
    finally:
        pkv.set_adaptive_splits(prev)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    eo, el = compare_fp8_with_oracle(case, pools, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    one_o, one_l = run_fp8(case, pools, num_splits=1)
    q, _, _, bt, sl = case.host_bits()
    rows = lambda idx: oracle.paged_decode_fp8(q, pools.k8, pools.v8, pools.ks, pools.vs, bt, sl, case.scale,
                                               select=[tuple(r) for r in idx])[0]
    split_straddle_check(out.float().cpu().numpy(), one_o.float().cpu().numpy(), rows)
    assert max_abs_diff(lse.cpu().numpy(), one_l.cpu().numpy()) <= SPLIT_TOL


@pytest.mark.parametrize("name", ["ragged", "long"])
def test_fp8_workloads_with_adaptive_splits(name):
    """Full-size workloads on the fp8 cache with the adaptive split count on: sampled rows against
    the fp8 oracle and the split-count bar against the planned split."""
    case = make_case(name)
    pools = Fp8Pools(case, poison_scales=False)
    dcase = case.to("cuda")
    base_o, base_l = run_fp8(dcase, pools)
    prev = pkv.set_adaptive_splits(True)
    try:
        out, lse = run_fp8(dcase, pools)
    finally:
        pkv.set_adaptive_splits(prev)
    eo, el = compare_fp8_with_oracle(case, pools, out, lse, select=sample_rows(case, n=16, seed=6))
    assert eo <= OUT_TOL and el <= LSE_TOL, (name, eo, el)
    assert max_abs_diff(lse.cpu().numpy(), base_l.cpu().numpy()) <= SPLIT_TOL
    q, _, _, bt, sl = case.host_bits()
    rows = lambda idx: oracle.paged_decode_fp8(q, pools.k8, pools.v8, pools.ks, pools.vs, bt, sl, case.scale,
                                               select=[tuple(r) for r in idx])[0]
    split_straddle_check(out.float().cpu().numpy(), base_o.float().cpu().numpy(), rows)
    del case, dcase, pools, out, lse, base_o, base_l
    torch.cuda.empty_cache()


@pytest.mark.parametrize("idx", [0, 1, 2], ids=["B65535", "G32-D256-P256", "G32-D128-P256"])
def test_fp8_maximum_sizes(idx):
    """The largest sizes the entry points take, on the fp8 cache, against the fp8 oracle in full."""
    from test_edges import MAXIMUM
    B, Hq, Hkv, D, P, lens = MAXIMUM[idx]
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B % 997 + D), seq_lens=lens, poison=True)
    pools = Fp8Pools(case)
    out, lse = run_fp8(case, pools)
    eo, el = compare_fp8_with_oracle(case, pools, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all()
