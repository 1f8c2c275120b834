"""Pins for the CPU fp64 oracle (no GPU).

The pages print no numeric attention example, so the oracle is pinned by what
the definition and the mathematics fix: hand-derived golden cases, single-token
rows, constant V, all-equal K, invariance to physical page placement and page
size, a brute-force comparison with torch's own float64 attention, merge
associativity, scale -> 0, the GQA mapping and poisoned padding.  Each pin is
chosen so that a plausible slip in the oracle (a dropped scale, exp vs exp2, a
wrong GQA index, a page off-by-one, a missing normaliser, a transposed operand,
no max subtraction) fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bits_to_bf16, make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _f(x):
    return float("-inf") if x == "-inf" else float(x)


def _bits(a):
    return bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def _run_case(c, **kw):
    q, k, v, bt, sl = c.host_bits()
    return oracle.paged_decode(q, k, v, bt, sl, c.scale, **kw)


def _dense(c):
    """Gather each sequence's K/V rows through the block table, with numpy indexing."""
    q, k, v, bt, sl = c.host_bits()
    kf = bits_to_bf16(k).double().numpy()
    vf = bits_to_bf16(v).double().numpy()
    seqs = []
    for b in range(c.B):
        L = int(sl[b])
        idx = np.arange(L)
        pages = bt[b, idx // c.P]
        slots = idx % c.P
        seqs.append((kf[pages, slots], vf[pages, slots]))  # [L, Hkv, D]
    return bits_to_bf16(q).double(), seqs


# --------------------------------------------------------------------------- golden


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["decode"], ids=lambda c: c["name"])
def test_golden_decode(case):
    P, Hq, Hkv, D, npg = case["P"], case["Hq"], case["Hkv"], case["D"], case["num_pages"]
    k = np.zeros((npg, P, Hkv, D), np.float32)
    v = np.zeros((npg, P, Hkv, D), np.float32)
    bt = np.asarray(case["block_table"], np.int32)
    L = case["seq_lens"][0]
    if "tokens" in case:
        for j in range(L):
            pg, sl = bt[0, j // P], j % P
            k[pg, sl, 0] = case["tokens"]["k"][j]
            v[pg, sl, 0] = case["tokens"]["v"][j]
    else:
        per = case["tokens_per_kv_head"]
        for g in range(Hkv):
            for j in range(L):
                pg, sl = bt[0, j // P], j % P
                k[pg, sl, g] = per["k"][g][j]
                v[pg, sl, g] = per["v"][g][j]
    out, lse = oracle.paged_decode(_bits(case["q"]), _bits(k), _bits(v), bt,
                                   np.asarray(case["seq_lens"], np.int32),
                                   np.float32(case["scale"]))
    exp_out = np.asarray(case["out"], np.float64)
    exp_lse = np.asarray([[_f(x) for x in row] for row in case["lse"]])
    assert np.max(np.abs(out - exp_out)) <= case["tol"]
    assert np.max(np.abs(lse - exp_lse)) <= case["tol"]


@pytest.mark.parametrize("case", _golden()["merge"], ids=lambda c: c["name"])
def test_golden_merge(case):
    po = np.asarray(case["partial_out"], np.float64)
    pl = np.asarray([[_f(x) for x in row] for row in case["partial_lse"]])
    out, lse = oracle.merge(po, pl)
    exp_lse = np.asarray([_f(x) for x in case["lse"]])
    assert np.max(np.abs(out - np.asarray(case["out"]))) <= case["tol"]
    fin = np.isfinite(exp_lse)
    assert np.all(np.isneginf(lse[~fin]))
    if fin.any():
        assert np.max(np.abs(lse[fin] - exp_lse[fin])) <= case["tol"]


# --------------------------------------------------------------------------- closed forms


def _spec(B=2, Hq=8, Hkv=2, D=64, P=16, pool=None, seed=0):
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), pool=pool, seed=seed)


def test_single_token_returns_v_row_exactly():
    # P-1: one key -> softmax weight exactly 1 -> out is that V row, lse is s_0.
    c = make_case(_spec(B=3, Hq=6, Hkv=3, D=64, P=8, pool=20), seq_lens=[1, 1, 1], poison=True)
    out, lse = _run_case(c)
    _, seqs = _dense(c)
    G = c.G
    for b in range(c.B):
        for h in range(c.Hq):
            assert np.array_equal(out[b, h], seqs[b][1][0, h // G])
    # lse = s_0 exactly when q and k are one-hot with exactly representable values.
    q = np.zeros((1, 1, 8), np.float32); q[0, 0, 3] = 1.5
    k = np.zeros((1, 8, 1, 8), np.float32); k[0, 0, 0, 3] = -2.75
    out, lse = oracle.paged_decode(_bits(q), _bits(k), _bits(k), np.zeros((1, 1), np.int32),
                                   np.asarray([1], np.int32), 0.125)
    assert lse[0, 0] == 0.125 * 1.5 * -2.75


def test_constant_v_returns_constant():
    # P-2: every used V row equals c -> out = c whatever the weights.
    c = make_case(_spec(B=2, Hq=8, Hkv=2, D=32, P=16), seq_lens=[37, 300], poison=True)
    crow = torch.randn(c.Hkv, c.D, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    v = c.v_cache.clone()
    bt = c.block_table.numpy()
    for b in range(c.B):
        for j in range(int(c.seq_lens[b])):
            v[bt[b, j // c.P], j % c.P] = crow
    c.v_cache = v
    out, _ = _run_case(c)
    for h in range(c.Hq):
        want = crow[h // c.G].double().numpy()
        assert np.allclose(out[:, h], want[None], rtol=1e-14, atol=1e-14)


def test_all_equal_k_gives_mean_of_v_and_log_length():
    # P-3: q = 0 -> every score is 0 -> out = mean_j v_j, lse = ln L.
    c = make_case(_spec(B=2, Hq=4, Hkv=1, D=16, P=8), seq_lens=[5, 77])
    c.q = torch.zeros_like(c.q)
    out, lse = _run_case(c)
    _, seqs = _dense(c)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        assert np.allclose(lse[b], math.log(L), rtol=0, atol=1e-14)
        mean = seqs[b][1][:, 0].mean(axis=0)
        assert np.allclose(out[b], mean[None], rtol=1e-13, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    # P-9: scale -> 0 flattens the softmax whatever q and K are.
    c = make_case(_spec(B=1, Hq=2, Hkv=2, D=16, P=16), seq_lens=[50], scale=0.0)
    out, lse = _run_case(c)
    _, seqs = _dense(c)
    for h in range(2):
        assert np.allclose(out[0, h], seqs[0][1][:, h].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert abs(lse[0, h] - math.log(50)) < 1e-14


def test_large_scores_do_not_overflow():
    # Scores near 1e3 would overflow exp() without the max subtraction.
    c = make_case(_spec(B=1, Hq=2, Hkv=1, D=64, P=16), seq_lens=[40], scale=40.0)
    out, lse = _run_case(c)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    assert lse.max() > 300  # the scores really are large
    _check_against_torch(c, out, lse, tol=1e-10)


def test_empty_sequence():
    c = make_case(_spec(B=3, Hq=4, Hkv=2, D=16, P=8), seq_lens=[0, 9, 0])
    out, lse = _run_case(c)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(lse[1]))


# --------------------------------------------------------------------------- invariances


def test_physical_page_invariance_bitwise():
    # P-5: the same logical K/V on two different page placements (and pool sizes).
    a = make_case(_spec(B=3, Hq=8, Hkv=2, D=64, P=16), seq_lens=[100, 1, 33], seed=11)
    q, k, v, bt, sl = a.host_bits()
    out_a, lse_a = oracle.paged_decode(q, k, v, bt, sl, a.scale)
    rng = np.random.default_rng(5)
    new_pool = a.num_pages + 9
    perm = rng.permutation(new_pool)[: a.num_pages]   # old page p -> new page perm[p]
    k2 = np.full((new_pool,) + k.shape[1:], 0x7FC0, np.uint16)   # NaN everywhere else
    v2 = np.full_like(k2, 0x7FC0)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(bt >= 0, perm[np.clip(bt, 0, None)], -1).astype(np.int32)
    out_b, lse_b = oracle.paged_decode(q, k2, v2, bt2, sl, a.scale)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_page_size_invariance_bitwise():
    # P-6: the same logical sequences repaged with P in {8, 16, 64}.
    _, seqs = None, None
    base = make_case(_spec(B=2, Hq=4, Hkv=2, D=32, P=8), seq_lens=[130, 64], seed=3)
    q, k, v, bt, sl = base.host_bits()
    results = []
    for P in (8, 16, 64):
        pages = [(int(L) + P - 1) // P for L in sl]
        npg = sum(pages) + 3
        k2 = np.full((npg, P, base.Hkv, base.D), 0x7FC0, np.uint16)
        v2 = np.full_like(k2, 0x7FC0)
        bt2 = np.full((base.B, max(pages)), -1, np.int32)
        nxt = npg - 1
        for b in range(base.B):
            for j in range(pages[b]):
                bt2[b, j] = nxt
                nxt -= 1
            for t in range(int(sl[b])):
                src_p, src_s = bt[b, t // base.P], t % base.P
                k2[bt2[b, t // P], t % P] = k[src_p, src_s]
                v2[bt2[b, t // P], t % P] = v[src_p, src_s]
        results.append(oracle.paged_decode(q, k2, v2, bt2, sl, base.scale))
    for o, l in results[1:]:
        assert np.array_equal(o, results[0][0]) and np.array_equal(l, results[0][1])


def test_poisoned_padding_is_ignored():
    # NaN in unused slots/pages and garbage table entries past the used pages.
    clean = make_case(_spec(B=2, Hq=8, Hkv=2, D=64, P=16), seq_lens=[45, 17], seed=4)
    dirty = make_case(_spec(B=2, Hq=8, Hkv=2, D=64, P=16), seq_lens=[45, 17], seed=4, poison=True)
    o1, l1 = _run_case(clean)
    o2, l2 = _run_case(dirty)
    assert np.all(np.isfinite(o2))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_thread_count_does_not_change_results():
    c = make_case(_spec(B=2, Hq=8, Hkv=2, D=64, P=16), seq_lens=[200, 3], seed=9)
    a = _run_case(c, nthreads=1)
    b = _run_case(c, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_selection_matches_full_run():
    c = make_case(_spec(B=3, Hq=8, Hkv=4, D=32, P=8), seq_lens=[10, 60, 7], seed=2)
    full_o, full_l = _run_case(c)
    pairs = [(2, 7), (0, 0), (1, 3)]
    o, l = _run_case(c, select=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(o[i], full_o[b, h]) and l[i] == full_l[b, h]


def test_bad_page_id_is_reported():
    c = make_case(_spec(B=1, Hq=2, Hkv=1, D=16, P=8), seq_lens=[20])
    c.block_table[0, 1] = c.num_pages + 5
    with pytest.raises(ValueError):
        _run_case(c)


# --------------------------------------------------------------------------- brute force


def _check_against_torch(c, out, lse, tol):
    q, seqs = _dense(c)
    G = c.G
    for b in range(c.B):
        kd = torch.from_numpy(seqs[b][0]).permute(1, 0, 2)  # [Hkv, L, D]
        vd = torch.from_numpy(seqs[b][1]).permute(1, 0, 2)
        kd = kd.repeat_interleave(G, dim=0)                   # contiguous GQA groups
        vd = vd.repeat_interleave(G, dim=0)
        qb = q[b].unsqueeze(1)                                # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qb, kd, vd, scale=float(np.float32(c.scale)))[:, 0]
        scores = (qb @ kd.transpose(1, 2))[:, 0] * float(np.float32(c.scale))
        ref_lse = torch.logsumexp(scores, dim=-1)
        assert np.max(np.abs(out[b] - ref.numpy())) <= tol
        assert np.max(np.abs(lse[b] - ref_lse.numpy())) <= tol


@pytest.mark.parametrize("D,Hq,Hkv,P,lens", [
    (8, 2, 1, 8, [1, 40, 13]),
    (64, 4, 2, 16, [33, 2]),
    (64, 4, 1, 8, [17]),
    (8, 8, 2, 4, [39, 16, 5]),
])
def test_brute_force_against_torch_float64(D, Hq, Hkv, P, lens):
    # P-7: an independent library routine on tiny inputs.
    c = make_case(dict(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, lens=("fixed", 1), seed=21),
                  seq_lens=lens, poison=True)
    out, lse = _run_case(c)
    _check_against_torch(c, out, lse, tol=1e-12)


def test_ragged_workload_sample_against_torch():
    # The ragged serving recipe (K rows scaled by U(0.5, 4): sharp softmax) on a few sequences.
    spec = dict(B=3, Hq=8, Hkv=2, D=64, P=16, lens=("fixed", 1), seed=8, k_row_scale=(0.5, 4.0))
    c = make_case(spec, seq_lens=[17, 250, 129])
    out, lse = _run_case(c)
    _check_against_torch(c, out, lse, tol=1e-12)


# --------------------------------------------------------------------------- merge


def test_merge_associativity():
    # P-8: merging the oracle's result over the first part and over the rest of the
    # keys gives the oracle's result over all keys.
    c = make_case(_spec(B=2, Hq=8, Hkv=2, D=32, P=16), seq_lens=[96, 160], seed=13)
    q, k, v, bt, sl = c.host_bits()
    full_o, full_l = oracle.paged_decode(q, k, v, bt, sl, c.scale)
    for cut_pages in (1, 2, 5):
        cut = cut_pages * c.P
        sl1 = np.minimum(sl, cut).astype(np.int32)
        o1, l1 = oracle.paged_decode(q, k, v, bt, sl1, c.scale)
        bt2 = np.full_like(bt, -1)
        bt2[:, : bt.shape[1] - cut_pages] = bt[:, cut_pages:]
        sl2 = np.maximum(sl - cut, 0).astype(np.int32)
        o2, l2 = oracle.paged_decode(q, k, v, bt2, sl2, c.scale)
        po = np.stack([o1.reshape(-1, c.D), o2.reshape(-1, c.D)])
        pl = np.stack([l1.reshape(-1), l2.reshape(-1)])
        mo, ml = oracle.merge(po, pl)
        assert np.max(np.abs(mo - full_o.reshape(-1, c.D))) <= 1e-12
        assert np.max(np.abs(ml - full_l.reshape(-1))) <= 1e-12


def test_merge_single_split_is_identity():
    rng = np.random.default_rng(0)
    po = rng.standard_normal((1, 5, 8))
    pl = rng.standard_normal((1, 5)) * 10
    o, l = oracle.merge(po, pl)
    assert np.array_equal(o, po[0]) and np.allclose(l, pl[0], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- kv append


def test_kv_append_hand_case():
    # P=4, two kv heads, D=2.  Sequence 0 appends key 5 -> logical page 1 (physical 1), slot 1;
    # sequence 1 appends key 0 -> logical page 0 (physical 0), slot 0.
    P, Hkv, D = 4, 2, 2
    k = np.zeros((4, P, Hkv, D), np.uint16)
    v = np.zeros_like(k)
    kn = np.arange(1, 9, dtype=np.uint16).reshape(2, Hkv, D)
    vn = kn + 100
    bt = np.array([[3, 1], [0, 2]], np.int32)
    k2, v2, rej = oracle.kv_append(kn, vn, bt, np.array([5, 0], np.int32), k, v)
    assert rej == 0
    want_k = np.zeros_like(k)
    want_k[1, 1] = kn[0]
    want_k[0, 0] = kn[1]
    assert np.array_equal(k2, want_k) and np.array_equal(v2, np.where(want_k > 0, want_k + 100, 0))
    assert np.array_equal(k, 0 * k)  # inputs untouched


def test_kv_append_skips_and_rejects():
    P, Hkv, D = 4, 1, 2
    k = np.full((3, P, Hkv, D), 7, np.uint16)
    kn = np.ones((3, Hkv, D), np.uint16)
    bt = np.array([[0, 1], [2, -1], [1, 0]], np.int32)
    k2, v2, rej = oracle.kv_append(kn, kn, bt, np.array([-1, 5, 8], np.int32), k, k)
    # -1: skipped silently; 5 -> logical page 1 holds -1 (bad id); 8 >= max_pages * P
    assert rej == 2 and np.array_equal(k2, k) and np.array_equal(v2, k)


def test_append_then_decode_matches_brute_force():
    # The appended key joins the softmax exactly as a key that was always there.
    c = make_case(_spec(B=3, Hq=8, Hkv=2, D=64, P=16), seq_lens=[16, 37, 0], seed=17)
    q, k, v, bt, sl = c.host_bits()
    g = torch.Generator().manual_seed(3)
    kn = bf16_bits(torch.randn(c.B, c.Hkv, c.D, generator=g).to(torch.bfloat16))
    vn = bf16_bits(torch.randn(c.B, c.Hkv, c.D, generator=g).to(torch.bfloat16))
    # sequence 0 is page-aligned (16 keys): its new key opens a new page
    bt = np.concatenate([bt, np.full((c.B, 1), -1, np.int32)], axis=1)
    spare = [c.num_pages, c.num_pages + 1, c.num_pages + 2]
    k = np.concatenate([k, np.zeros((3,) + k.shape[1:], np.uint16)])
    v = np.concatenate([v, np.zeros((3,) + v.shape[1:], np.uint16)])
    for b in range(c.B):
        bt[b, int(sl[b]) // c.P] = spare[b] if int(sl[b]) % c.P == 0 else bt[b, int(sl[b]) // c.P]
    k2, v2, rej = oracle.kv_append(kn, vn, bt, sl, k, v)
    assert rej == 0
    out, lse = oracle.paged_decode(q, k2, v2, bt, sl + 1, c.scale)
    qf = bits_to_bf16(q).double()
    kf = bits_to_bf16(k2).double().numpy()
    vf = bits_to_bf16(v2).double().numpy()
    for b in range(c.B):
        idx = np.arange(int(sl[b]) + 1)
        kd = torch.from_numpy(kf[bt[b, idx // c.P], idx % c.P]).permute(1, 0, 2).repeat_interleave(c.G, 0)
        vd = torch.from_numpy(vf[bt[b, idx // c.P], idx % c.P]).permute(1, 0, 2).repeat_interleave(c.G, 0)
        # the last key/value rows are the appended ones
        assert np.array_equal(kd[:, -1].numpy(), bits_to_bf16(kn[b]).double().numpy().repeat(c.G, 0))
        ref = torch.nn.functional.scaled_dot_product_attention(qf[b].unsqueeze(1), kd, vd, scale=c.scale)[:, 0]
        assert np.max(np.abs(out[b] - ref.numpy())) <= 1e-12
