"""Pins for the oracle's multi-token rows (no GPU): several query rows per request,
ragged by qo_indptr, with or without the causal mask aligned to the end of the keys.

Each pin ties the new entry point to something independent of it: the single-row
decode oracle (one row per request, a truncated length for the causal rows, each row
as its own request), torch's float64 attention with an explicit mask, and the
definition's special cases (rows that see no key, the fp8 cache), and hand-derived cases
(tests/golden/hand_cases.json, "prefill")."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bits_to_bf16, make_case, make_prefill_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _golden_prefill():
    with open(GOLDEN) as f:
        return json.load(f)["prefill"]


def _bits(a):
    return bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def _num(x):
    return float("-inf") if x == "-inf" else float(x)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("case", _golden_prefill(), ids=lambda c: c["name"])
def test_golden_prefill(case, causal):
    P, Hkv, D, npg = case["P"], case["Hkv"], case["D"], case["num_pages"]
    k = np.zeros((npg, P, Hkv, D), np.float32)
    v = np.zeros((npg, P, Hkv, D), np.float32)
    for pg, rows in case["pages"].items():
        for slot, (kr, vr) in enumerate(zip(rows["k"], rows["v"])):
            k[int(pg), slot] = kr
            v[int(pg), slot] = vr
    scale = float(np.float32(case["scale"]))  # the C interface passes the scale as a float32
    out, lse = oracle.paged_prefill(_bits(case["q"]), np.asarray(case["qo_indptr"], np.int32),
                                    np.asarray(case["block_table"], np.int32), np.asarray(case["seq_lens"], np.int32),
                                    scale, causal=causal, k_bits=_bits(k), v_bits=_bits(v))
    want = case["causal" if causal else "noncausal"]
    want_out = np.asarray(want["out"], np.float64)
    want_lse = np.vectorize(_num)(np.asarray(want["lse"], dtype=object)).astype(np.float64)
    assert np.abs(out - want_out).max() <= case["tol"] + 1e-12
    inf = np.isinf(want_lse)
    assert np.array_equal(np.isneginf(lse), inf)
    assert np.abs(lse[~inf] - want_lse[~inf]).max() <= case["tol"] + 1e-12


def _spec(B, Hq, Hkv, D, P, seed=0):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=seed)


def _host(c):
    q, k, v, bt, sl = c.host_bits()
    return q, k, v, bt, sl, c.qo_indptr.cpu().numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_one_row_per_request_is_decode(causal):
    c = make_prefill_case(_spec(3, 8, 2, 64, 16, seed=1), q_lens=[1, 1, 1], kv_lens=[1, 40, 200])
    q, k, v, bt, sl, qo = _host(c)
    o1, l1 = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=causal, k_bits=k, v_bits=v)
    o2, l2 = oracle.paged_decode(q, k, v, bt, sl, c.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_row_is_decode_over_its_visible_prefix():
    c = make_prefill_case(_spec(2, 8, 2, 64, 16, seed=2), q_lens=[5, 3], kv_lens=[37, 3])
    q, k, v, bt, sl, qo = _host(c)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=True, k_bits=k, v_bits=v)
    for b in range(2):
        n = qo[b + 1] - qo[b]
        for i in range(n):
            t = qo[b] + i
            visible = sl[b] - n + i + 1
            do, dl = oracle.paged_decode(q[t:t + 1], k, v, bt[b:b + 1], np.array([visible], np.int32), c.scale)
            assert np.array_equal(out[t], do[0]) and np.array_equal(lse[t], dl[0])


def test_non_causal_row_is_decode_over_all_keys():
    c = make_prefill_case(_spec(2, 16, 4, 128, 8, seed=3), q_lens=[4, 2], kv_lens=[50, 9])
    q, k, v, bt, sl, qo = _host(c)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=False, k_bits=k, v_bits=v)
    for t in range(qo[-1]):
        b = int(np.searchsorted(qo, t, side="right") - 1)
        do, dl = oracle.paged_decode(q[t:t + 1], k, v, bt[b:b + 1], sl[b:b + 1], c.scale)
        assert np.array_equal(out[t], do[0]) and np.array_equal(lse[t], dl[0])


@pytest.mark.parametrize("q_lens,kv_lens,G", [([3, 1, 6], [10, 1, 33], 4), ([8, 2], [8, 20], 2), ([4], [4], 1)])
def test_brute_force_against_torch_float64_with_an_explicit_mask(q_lens, kv_lens, G):
    Hkv, D, P = 2, 64, 4
    c = make_prefill_case(_spec(len(q_lens), Hkv * G, Hkv, D, P, seed=4), q_lens=q_lens, kv_lens=kv_lens)
    q, k, v, bt, sl, qo = _host(c)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=True, k_bits=k, v_bits=v)
    kf, vf = bits_to_bf16(k).double(), bits_to_bf16(v).double()
    qf = bits_to_bf16(q).double()
    for b, (n, L) in enumerate(zip(q_lens, kv_lens)):
        idx = torch.arange(L)
        pages = torch.from_numpy(bt[b])[idx // P].long()
        K = kf[pages, idx % P].repeat_interleave(G, dim=1).permute(1, 0, 2)  # [Hq, L, D]
        V = vf[pages, idx % P].repeat_interleave(G, dim=1).permute(1, 0, 2)
        Q = qf[qo[b]:qo[b + 1]].permute(1, 0, 2)                             # [Hq, n, D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=c.scale)
        s = torch.einsum("hnd,hld->hnl", Q, K) * c.scale
        ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        assert np.allclose(out[qo[b]:qo[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        assert np.allclose(lse[qo[b]:qo[b + 1]], ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_rows_that_see_no_key():
    # 5 query rows over 3 keys: the first two rows see nothing under the causal mask
    c = make_prefill_case(_spec(1, 4, 1, 64, 8, seed=5), q_lens=[5], kv_lens=[3])
    q, k, v, bt, sl, qo = _host(c)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=True, k_bits=k, v_bits=v)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:2])) and np.all(np.isfinite(lse[2:]))
    # an empty request in the middle owns no row
    c2 = make_prefill_case(_spec(3, 4, 1, 64, 8, seed=6), q_lens=[2, 0, 1], kv_lens=[9, 4, 5])
    q, k, v, bt, sl, qo = _host(c2)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c2.scale, causal=True, k_bits=k, v_bits=v)
    assert out.shape[0] == 3 and np.all(np.isfinite(lse))


def test_fp8_cache_matches_the_fp8_decode_row_by_row():
    c = make_prefill_case(_spec(2, 8, 2, 128, 16, seed=7), q_lens=[3, 2], kv_lens=[40, 17])
    q, k, v, bt, sl, qo = _host(c)
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    out, lse = oracle.paged_prefill(q, qo, bt, sl, c.scale, causal=True, fp8=(k8, v8, ks, vs))
    for b in range(2):
        n = qo[b + 1] - qo[b]
        for i in range(n):
            t = qo[b] + i
            do, dl = oracle.paged_decode_fp8(q[t:t + 1], k8, v8, ks, vs, bt[b:b + 1],
                                             np.array([sl[b] - n + i + 1], np.int32), c.scale)
            assert np.array_equal(out[t], do[0]) and np.array_equal(lse[t], dl[0])


def test_selection_matches_full_run_and_bad_indptr_is_rejected():
    c = make_prefill_case(_spec(2, 8, 2, 64, 16, seed=8), q_lens=[3, 4], kv_lens=[20, 30])
    q, k, v, bt, sl, qo = _host(c)
    full_o, full_l = oracle.paged_prefill(q, qo, bt, sl, c.scale, k_bits=k, v_bits=v)
    rows = [(0, 0), (6, 7), (3, 2)]
    o, l = oracle.paged_prefill(q, qo, bt, sl, c.scale, k_bits=k, v_bits=v, select=rows)
    for n, (t, h) in enumerate(rows):
        assert np.array_equal(o[n], full_o[t, h]) and l[n] == full_l[t, h]
    with pytest.raises(ValueError):
        oracle.paged_prefill(q, np.array([0, 3, 6], np.int32), bt, sl, c.scale, k_bits=k, v_bits=v)
