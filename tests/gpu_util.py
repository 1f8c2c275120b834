"""Helpers shared by the GPU tests: run the CUDA path through the C-ABI binding
and compare it with the CPU oracle."""
import numpy as np
import torch

import oracle
import paged_kv_gqa_gb300 as pkv

OUT_TOL = 1.5e-2     # max |out_gpu - out_oracle| on bf16 outputs
LSE_TOL = 1e-3       # max |lse_gpu - lse_oracle| on f32 LSE
SPLIT_TOL = 2e-3     # max |out(S1) - out(S2)| between split counts


def run_gpu(case, num_splits=0, with_lse=True, expect_status=0):
    """One call of paged_decode_attn_ex on the case's tensors (moved to cuda:0)."""
    c = case if case.q.is_cuda else case.to("cuda")
    ws_bytes = pkv.paged_decode_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages,
                                                    num_splits=num_splits)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    pkv.paged_decode_attn_ex(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale, out, lse, ws,
                             num_splits=num_splits)
    status = pkv.pkv_check_status(ws)
    assert status == expect_status, "device status %s" % pkv.STATUS.get(status, status)
    return out, lse


def max_abs_diff(a, b):
    """max |a - b| where equal infinities count as 0."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    return float(np.max(d)) if d.size else 0.0


def compare_with_oracle(case, out, lse, select=None, nthreads=0):
    """Returns (max out error, max lse error) against the oracle (all rows or a sample)."""
    q, k, v, bt, sl = case.host_bits()
    ref_o, ref_l = oracle.paged_decode(q, k, v, bt, sl, case.scale, select=select, nthreads=nthreads)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy() if lse is not None else None
    if select is not None:
        idx = np.asarray(list(select))
        o = o[idx[:, 0], idx[:, 1]]
        l = l[idx[:, 0], idx[:, 1]] if l is not None else None
    eo = max_abs_diff(o, ref_o)
    el = max_abs_diff(l, ref_l) if l is not None else 0.0
    return eo, el


def sample_rows(case, n=24, seed=0):
    """A seeded sample of (b, h) rows, always including the longest and the shortest sequence."""
    rng = np.random.default_rng(seed)
    lens = case.seq_lens.cpu().numpy()
    rows = {(int(np.argmax(lens)), 0), (int(np.argmax(lens)), case.Hq - 1), (int(np.argmin(lens)), case.Hq // 2),
            (0, 0), (case.B - 1, case.Hq - 1)}
    while len(rows) < n:
        rows.add((int(rng.integers(case.B)), int(rng.integers(case.Hq))))
    return sorted(rows)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    x = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(x)) - 7)


def split_invariance_violation(a, b, tol=SPLIT_TOL):
    """Largest excess of |a - b| over the split-count bar.

    Different split counts only reorder f32 sums, so the f32 results agree to
    far better than 2e-3; after rounding to bf16 two such values may still land
    one rounding step apart when they straddle a rounding boundary.  An element
    passes when it is within `tol` or within one bf16 step of the larger value.
    Returns (max excess, fraction of elements that differ at all, max |a-b|)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.abs(a - b)
    allowed = np.maximum(tol, bf16_ulp(np.maximum(np.abs(a), np.abs(b))))
    return float(np.max(d - allowed)), float(np.mean(d > 0)), float(np.max(d))


def bf16_adjacent(a, b):
    """True where a and b (float arrays holding bf16 values) are neighbouring bf16 numbers:
    the same sign and bit patterns one apart."""
    ia = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    ib = torch.from_numpy(np.ascontiguousarray(b, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    same_sign = (ia < 0) == (ib < 0)
    return same_sign & (np.abs(ia.astype(np.int32) - ib.astype(np.int32)) == 1)


def split_straddle_check(a, b, oracle_rows, tol=SPLIT_TOL, out_tol=OUT_TOL):
    """The split-count bar on bf16 outputs, with every element past it proved a rounding straddle.

    a, b: outputs of the same call at two split counts, float arrays [rows..., D] of bf16
    values.  Split counts only reorder f32 sums, so where |a - b| > tol the two f32 results
    must have straddled a bf16 rounding boundary.  Each such element must therefore be
      (i)   one bf16 step: a and b neighbouring bf16 numbers;
      (ii)  a genuine straddle: the fp64 oracle value lies within tol of the midpoint of a and b
            (the rounding boundary both f32 sums sat beside);
      (iii) within out_tol of the oracle on both sides.
    oracle_rows(idx) returns the fp64 oracle outputs [n, D] for the row indices idx ([n, ndim-1]).
    Returns (number of elements past tol, max |a - b|, max |oracle - midpoint| over them); raises
    AssertionError naming the first element that breaks (i)-(iii)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.abs(a - b)
    big = d > tol
    n_big = int(big.sum())
    if n_big == 0:
        return 0, float(d.max()) if d.size else 0.0, 0.0
    lead = np.argwhere(big)[:, :-1]
    rows = np.unique(lead, axis=0)
    ref = np.asarray(oracle_rows(rows), np.float64).reshape(len(rows), a.shape[-1])
    pos = {tuple(r): i for i, r in enumerate(rows.tolist())}
    worst_mid = 0.0
    for e in np.argwhere(big):
        r, col = tuple(e[:-1].tolist()), int(e[-1])
        x, y, o = a[tuple(e)], b[tuple(e)], ref[pos[r], col]
        assert bf16_adjacent(np.array([x]), np.array([y]))[0], ("not one bf16 step", r, col, x, y)
        mid = 0.5 * (x + y)
        worst_mid = max(worst_mid, abs(o - mid))
        assert abs(o - mid) <= tol, ("not a rounding straddle", r, col, x, y, o)
        assert abs(x - o) <= out_tol and abs(y - o) <= out_tol, ("past the oracle bar", r, col, x, y, o)
    return n_big, float(d.max()), worst_mid


def decode_oracle_rows(case):
    """oracle_rows for split_straddle_check on a decode case: (b, h) rows -> fp64 outputs."""
    q, k, v, bt, sl = case.host_bits()
    return lambda rows: oracle.paged_decode(q, k, v, bt, sl, case.scale, select=[tuple(r) for r in rows])[0]
