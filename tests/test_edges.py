"""Edge cases of the CUDA path against the CPU oracle, through the C-ABI.

Each case targets a place where a plausible kernel mistake would hide from the
workload tests: a sharply peaked softmax (running maxima that jump by tens of
units, deferred rescaling on the tensor-core path), a zero or negative scale
(uniform and inverted weights), the largest group size at the largest head
dimension, a forced single split longer than one block's block-table slice, and the
largest sizes the entry points take (65535 sequences, G = 32 with 256-key pages).
Bars as everywhere: max |out - oracle| <= 1.5e-2, max |lse - oracle| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, compare_with_oracle, run_gpu
from workloads import make_case, make_prefill_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _spec(B, Hq, Hkv, D, P, seed=0):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed)


# Scores with a standard deviation of about 8 (natural-log units): over a few thousand
# keys the largest beats the runner-up by several units, so each output is close to a
# single V row and the running maximum moves by large steps as the keys stream.
PEAKED = [
    # B, Hq, Hkv, D, P, lens
    (3, 32, 8, 128, 16, [3000, 17, 700]),
    (2, 8, 2, 64, 8, [1000, 4096]),
    (2, 32, 2, 256, 64, [2048, 100]),
]


# 20 splits: the in-kernel merge takes them eight at a time, so the running maximum moves
# between batches (and rescales what the earlier batches summed)
@pytest.mark.parametrize("splits", [1, 0, 7, 20])
@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", PEAKED, ids=lambda x: str(x).replace(" ", ""))
def test_peaked_softmax(B, Hq, Hkv, D, P, lens, splits):
    scale = 8.0 / math.sqrt(D)
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=11 + D), seq_lens=lens, poison=True, scale=scale)
    out, lse = run_gpu(case, num_splits=splits)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("scale", [0.0, -0.125])
def test_zero_and_negative_scale(scale):
    """scale 0 weights every key equally (lse = ln L); a negative scale inverts the weights."""
    lens = [1, 250, 3001]
    case = make_case(_spec(3, 16, 4, 128, 16, seed=21), seq_lens=lens, poison=True, scale=scale)
    for splits in (1, 0):
        out, lse = run_gpu(case, num_splits=splits)
        eo, el = compare_with_oracle(case, out, lse)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)
        if scale == 0.0:
            want = torch.tensor([math.log(L) for L in lens], dtype=torch.float64)
            assert (lse.double().cpu() - want[:, None]).abs().max().item() <= LSE_TOL


def test_group_32_at_head_dim_256():
    """G = 32 at D = 256: a block there serves at most 16 heads, so each group is two query tiles
    (the several-rows variant with one row per sequence), each merging its own splits."""
    case = make_case(_spec(2, 64, 2, 256, 16, seed=23), seq_lens=[1500, 33], poison=True)
    plan = pkv.plan_query(2, 64, 2, 256, 16, case.max_pages, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["q_tiles"] == 2 and plan["rows_per_block"] == 16, plan
    for splits in (1, 0, 3, 20):
        out, lse = run_gpu(case, num_splits=splits)
        eo, el = compare_with_oracle(case, out, lse)
        assert eo <= OUT_TOL and el <= LSE_TOL, (splits, eo, el)


def test_single_split_longer_than_a_table_slice():
    """One split asked for, but the sequence has more pages than a block stages: the plan
    must cap the chunk (two splits here) and the result must still be the whole softmax."""
    L = 70000
    case = make_case(_spec(1, 4, 1, 64, 16, seed=29), seq_lens=[L], poison=True)
    plan = pkv.plan_query(1, 4, 1, 64, 16, case.max_pages, 152, num_splits=1)
    assert plan["num_splits"] >= 2 and plan["chunk_tokens"] * plan["num_splits"] >= L
    out, lse = run_gpu(case, num_splits=1)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def _prefill(case, mode, causal=True):
    c = case.to("cuda")
    total_q = c.q.shape[0]
    mq = int(np.diff(case.qo_indptr.cpu().numpy()).max())
    ws = torch.zeros(pkv.paged_prefill_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, total_q, mq),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((total_q, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((total_q, c.Hq), float("nan"), dtype=torch.float32, device="cuda")
    prev = pkv.set_prefill_tensor_cores(mode)
    try:
        pkv.paged_prefill_attn(c.q, c.k_cache, c.v_cache, c.qo_indptr, c.block_table, c.seq_lens, mq, c.scale,
                               out, lse, ws, causal=causal)
    finally:
        pkv.set_prefill_tensor_cores(prev)
    assert pkv.pkv_check_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("mode", ["always", "rows128", "off"])
def test_peaked_softmax_several_rows(mode):
    """Several query rows per sequence with a peaked softmax: the tensor-core kernels let the
    reference maximum lag the true one by up to 2^8 before rescaling, so probabilities above
    1 reach the bf16 P operand; the result must still match the oracle."""
    import oracle
    case = make_prefill_case(_spec(2, 32, 4, 128, 16, seed=31), q_lens=[40, 17], kv_lens=[2000, 300],
                             poison=True, scale=8.0 / math.sqrt(128))
    out, lse = _prefill(case, mode)
    q, k, v, bt, sl = case.host_bits()
    ro, rl = oracle.paged_prefill(q, case.qo_indptr.cpu().numpy(), bt, sl, case.scale, causal=True,
                                  k_bits=k, v_bits=v)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.abs(o - ro).max() <= OUT_TOL and np.abs(l - rl).max() <= LSE_TOL


# The largest sizes the entry points take: 65535 sequences (the grid's z dimension), the
# largest group (G = 32) at the largest head dimension and page size.
MAXIMUM = [
    # B, Hq, Hkv, D, P, lens
    (65535, 4, 1, 64, 8, [(7 * i) % 23 for i in range(65535)]),
    (1, 32, 1, 256, 256, [6000]),
    (2, 32, 1, 128, 256, [20000, 1]),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,P,lens", MAXIMUM, ids=["B65535", "G32-D256-P256", "G32-D128-P256"])
def test_maximum_sizes(B, Hq, Hkv, D, P, lens):
    case = make_case(_spec(B, Hq, Hkv, D, P, seed=B % 1000 + D), seq_lens=lens, poison=True)
    out, lse = run_gpu(case)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    assert torch.isfinite(out.float()).all()


def test_batch_past_the_grid_limit_is_rejected():
    """65536 sequences: refused on the host with PKV_ERR_UNSUPPORTED before any launch (the
    outputs keep their sentinel)."""
    case = make_case(_spec(65536, 4, 1, 64, 8, seed=3), seq_lens=[1] * 65536).to("cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.full((case.B, case.Hq, case.D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((case.B, case.Hq), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError) as err:
        pkv.paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale, out,
                              lse, ws)
    assert err.value.status == -2
    torch.cuda.synchronize()
    assert bool((out.float() == 7.0).all()) and bool((lse == 7.0).all())
