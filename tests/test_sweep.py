"""A seeded sweep of random decode shapes on both caches, each checked in full against the oracle.

Each case draws a batch size, a group size (1-32), a head dim, a page size, sequence lengths
(empty ones, one-key ones, page-boundary ones and long ones) and a forced split count, so the
planner's tilings, the masked stage tails and the in-kernel merge (one batch of splits or
several) meet shapes no hand-picked case names.  Bars: max |out - oracle| <= 1.5e-2, max
|lse - oracle| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, compare_with_oracle, max_abs_diff, run_gpu
from workloads import make_case, used_slot_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128, 256]))
    G = int(rng.choice([1, 2, 3, 4, 8, 12, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4]))
    P = int(rng.choice([8, 16, 32, 64, 128, 256]))
    B = int(rng.integers(1, 9))
    kinds = rng.integers(0, 5, size=B)
    lens = []
    for k in kinds:
        if k == 0:
            lens.append(0)
        elif k == 1:
            lens.append(1)
        elif k == 2:
            lens.append(int(P * rng.integers(1, 6)))            # a whole number of pages
        elif k == 3:
            lens.append(int(rng.integers(2, 700)))
        else:
            lens.append(int(rng.integers(700, 6000)))
    splits = int(rng.choice([0, 1, 2, 5, 9, 17, 40]))
    return dict(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed), lens, splits


SEEDS = list(range(24))


@pytest.mark.parametrize("seed", SEEDS)
def test_random_shapes_bf16(seed):
    spec, lens, splits = _draw(seed)
    case = make_case(spec, seq_lens=lens, poison=True)
    out, lse = run_gpu(case, num_splits=splits)
    eo, el = compare_with_oracle(case, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL, (spec, lens, splits, eo, el)
    empty = [b for b, L in enumerate(lens) if L == 0]
    if empty:
        assert out[empty].float().abs().max().item() == 0 and torch.isneginf(lse[empty]).all()


@pytest.mark.parametrize("seed", SEEDS[::2])
def test_random_shapes_fp8(seed):
    spec, lens, splits = _draw(seed)
    case = make_case(spec, seq_lens=lens, poison=True)
    q, k, v, bt, sl = case.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    unused = ~used_slot_mask(case)
    for sc in (ks, vs):
        sc.transpose(0, 2, 1)[unused] = np.nan
    c = case.to("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = torch.zeros(pkv.paged_decode_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages,
                                                          num_splits=splits, cache="fp8"),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_decode_attn_fp8(c.q, t(k8), t(v8), t(ks), t(vs), c.block_table, c.seq_lens, c.scale, out, lse, ws,
                              num_splits=splits)
    assert pkv.pkv_check_status(ws) == 0
    ro, rl = oracle.paged_decode_fp8(q, k8, v8, ks, vs, bt, sl, case.scale)
    eo = max_abs_diff(out.float().cpu().numpy(), ro)
    el = max_abs_diff(lse.cpu().numpy(), rl)
    assert eo <= OUT_TOL and el <= LSE_TOL, (spec, lens, splits, eo, el)
