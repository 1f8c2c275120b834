"""Paged KV append on the GPU (through the C-ABI) against the CPU oracle.

Byte and index work: the pools after the append must equal the oracle's bit for
bit, everywhere (the written rows and every untouched byte, NaN padding included).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, compare_with_oracle, run_gpu
from workloads import Case, bf16_bits, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _append_case(B, Hq, Hkv, D, P, lens, seed):
    """A case whose table has room for one more key per sequence (a fresh page where
    the sequence ends on a page boundary), plus the new rows to append."""
    c = make_case(dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed), seq_lens=lens, poison=True)
    lens = np.asarray(lens)
    need_new = [b for b in range(B) if lens[b] % P == 0]
    extra = len(need_new)
    bt = c.block_table.numpy()
    bt = np.concatenate([bt, np.full((B, 1), -1, np.int32)], axis=1)
    for i, b in enumerate(need_new):
        bt[b, lens[b] // P] = c.num_pages + i
    nan = torch.full((extra,) + tuple(c.k_cache.shape[1:]), float("nan"), dtype=torch.bfloat16)
    c.k_cache = torch.cat([c.k_cache, nan])
    c.v_cache = torch.cat([c.v_cache, nan.clone()])
    c.num_pages += extra
    c.max_pages += 1
    c.block_table = torch.from_numpy(bt)
    g = torch.Generator().manual_seed(seed + 99)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    return c, kn, vn


def _gpu_append(c, kn, vn, positions, status=None):
    kc = c.k_cache.cuda()
    vc = c.v_cache.cuda()
    pkv.paged_kv_append(kn.cuda(), vn.cuda(), c.block_table.cuda(), torch.as_tensor(positions, dtype=torch.int32).cuda(),
                        kc, vc, status=status)
    torch.cuda.synchronize()
    return kc.cpu(), vc.cpu()


@pytest.mark.parametrize("B,Hkv,D,P,lens", [
    (3, 2, 64, 8, [0, 7, 8]),
    (4, 8, 128, 16, [15, 16, 17, 300]),
    (2, 2, 256, 64, [63, 64]),
    (300, 1, 128, 16, [(13 * i) % 70 for i in range(300)]),
], ids=lambda x: str(x).replace(" ", "")[:40])
def test_append_bit_exact(B, Hkv, D, P, lens):
    c, kn, vn = _append_case(B, Hkv * 2, Hkv, D, P, lens, seed=B + D)
    pos = np.asarray(lens, np.int32)
    if B > 2:
        pos[1] = -1  # a sequence with nothing to append this step
    kc, vc = _gpu_append(c, kn, vn, pos)
    rk, rv, rej = oracle.kv_append(bf16_bits(kn), bf16_bits(vn), c.block_table.numpy(), pos,
                                   bf16_bits(c.k_cache), bf16_bits(c.v_cache))
    assert rej == 0
    assert np.array_equal(bf16_bits(kc), rk) and np.array_equal(bf16_bits(vc), rv)


def test_append_reports_bad_positions_and_pages():
    c, kn, vn = _append_case(3, 4, 2, 128, 16, [20, 5, 9], seed=7)
    bt = c.block_table.numpy().copy()
    bt[2, 0] = c.num_pages + 3  # sequence 2's page id is out of range
    c.block_table = torch.from_numpy(bt)
    for pos, want in (([20, c.max_pages * 16, -1], -8), ([20, -1, 9], -6)):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kc, vc = _gpu_append(c, kn, vn, pos, status=status)
        assert int(status.item()) == want
        rk, rv, rej = oracle.kv_append(bf16_bits(kn), bf16_bits(vn), bt, np.asarray(pos, np.int32),
                                       bf16_bits(c.k_cache), bf16_bits(c.v_cache))
        assert rej == 1
        assert np.array_equal(bf16_bits(kc), rk) and np.array_equal(bf16_bits(vc), rv)


def test_append_then_decode():
    # One serving step: append the new token's K/V, then decode over L + 1 keys.
    c, kn, vn = _append_case(4, 32, 8, 128, 16, [31, 32, 1000, 1], seed=11)
    lens = c.seq_lens.numpy()
    kc, vc = _gpu_append(c, kn, vn, lens)
    stepped = Case(**c.__dict__)
    stepped.k_cache, stepped.v_cache = kc, vc
    stepped.seq_lens = torch.from_numpy((lens + 1).astype(np.int32))
    out, lse = run_gpu(stepped)
    eo, el = compare_with_oracle(stepped, out, lse)
    assert eo <= OUT_TOL and el <= LSE_TOL
