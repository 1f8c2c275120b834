"""Pins for the oracle's FP8 (e4m3) KV variant (no GPU).

The codec is pinned to the format's definition (hand-listed code values), to an
independent implementation (torch's float8_e4m3fn conversions) and to a brute-force
nearest-value search; the quantiser to its scale rule at the boundaries and to the
format's rounding-error bound; the fp8 decode to the bf16 decode of the same values
and to a hand-placed case whose scales sit at known (page, head, slot) positions.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, make_case


def _bits(a):
    return bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


# ------------------------------------------------------------------ codec

@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x0F, 1.875 * 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3C, 1.5), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9)),
])
def test_e4m3_values_from_the_format(code, value):
    assert oracle.e4m3_value([code])[0] == value


def test_e4m3_nan_and_negative_zero():
    v = oracle.e4m3_value([0x7F, 0xFF, 0x80])
    assert np.isnan(v[0]) and np.isnan(v[1])
    assert v[2] == 0.0 and math.copysign(1.0, v[2]) == -1.0


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ours = oracle.e4m3_value(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], ours[fin])
    assert np.array_equal(np.signbit(ref[fin]), np.signbit(ours[fin]))


def test_e4m3_encode_matches_torch_within_range():
    g = np.random.default_rng(5)
    mags = np.concatenate([g.uniform(0, 448, 3000), 2.0 ** g.uniform(-14, 8.8, 3000), g.uniform(0, 2 ** -6, 1000)])
    x = (mags * g.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_encode_is_the_nearest_code_ties_to_even():
    # brute force over the finite codes, independent of the encoder's bisection
    table = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    g = np.random.default_rng(9)
    mids = (table[:-1] + table[1:]) / 2  # exact ties
    x = np.concatenate([g.uniform(0, 448, 2000), mids, table])
    got = oracle.e4m3_encode(x)
    for xi, c in zip(x, got):
        d = np.abs(table - xi)
        best = np.flatnonzero(d == d.min())
        want = best[0] if best.size == 1 else best[best % 2 == 0][0]
        assert c == want, (xi, c, want)


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38), (1.1875, 0x3A), (7.5 * 2.0 ** -9, 0x08), (2.0 ** -10, 0x00), (2.0 ** -10 * 1.0001, 0x01),
    (448.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E), (-1e30, 0xFE), (float("-inf"), 0xFE),
    (float("nan"), 0x7F), (-0.0, 0x80), (-1e-30, 0x80), (0.0, 0x00),
])
def test_e4m3_encode_special_cases(x, code):
    assert oracle.e4m3_encode([x])[0] == code


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_value(codes)), codes)


# ------------------------------------------------------------------ quantiser

@pytest.mark.parametrize("amax,scale", [
    (448.0, 1.0), (450.0, 2.0), (1.0, 2.0 ** -8), (0.875, 2.0 ** -9), (0.0, 2.0 ** -64), (1e30, 2.0 ** 64),
    (2.0 ** -70, 2.0 ** -64), (3.0, 2.0 ** -7),
])
def test_quantizer_scale_rule(amax, scale):
    row = np.zeros((1, 64), np.float32)
    row[0, 5] = -amax
    row[0, 9] = amax / 4
    codes, scales = oracle.fp8_quantize_rows(_bits(row))
    assert scales[0] == np.float32(scale)
    # the scale is the smallest power of two that does not saturate the row
    if 0 < amax <= 448 * 2.0 ** 64 and scale > 2.0 ** -64:
        assert amax <= 448 * scale and amax > 448 * scale / 2


def test_quantizer_error_bound_and_tight_scale():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(512, 128, generator=g) * torch.exp2(torch.randint(-12, 12, (512, 1), generator=g).float())
    bits = bf16_bits(x.to(torch.bfloat16))
    codes, scales = oracle.fp8_quantize_rows(bits)
    xv = x.to(torch.bfloat16).double().numpy()
    deq = oracle.e4m3_value(codes) * scales[:, None].astype(np.float64)
    s = scales[:, None].astype(np.float64)
    # round to nearest with 3 mantissa bits: half an ulp is <= 2^-4 |x| for normals, 2^-10 s below 2^-6 s
    assert np.all(np.abs(deq - xv) <= np.maximum(2.0 ** -4 * np.abs(xv), 2.0 ** -10 * s))
    amax = np.abs(xv).max(axis=1)
    assert np.all(amax <= 448 * scales) and np.all(amax > 224 * scales)
    assert np.all(np.log2(scales) == np.round(np.log2(scales)))  # powers of two


def test_quantizer_nan_is_left_out_of_the_scale():
    row = np.full((1, 64), 2.0, np.float32)
    row[0, 3] = np.nan
    codes, scales = oracle.fp8_quantize_rows(_bits(row))
    assert scales[0] == np.float32(2.0 ** -7) and codes[0, 3] == 0x7F and codes[0, 0] == 0x78  # 2 / 2^-7 = 256 = 1.0 * 2^8


# ------------------------------------------------------------------ fp8 decode

def test_fp8_decode_equals_bf16_decode_on_the_dequantised_pool():
    c = make_case(dict(B=3, Hq=8, Hkv=2, D=64, P=16, lens=("fixed", 1), seed=4), seq_lens=[1, 37, 200])
    q, k, v, bt, sl = c.host_bits()
    k8, ks = oracle.quantize_pool(k)
    v8, vs = oracle.quantize_pool(v)
    kd, vd = oracle.dequantize_pool(k8, ks), oracle.dequantize_pool(v8, vs)
    # power-of-two scales: every dequantised value is an exact bf16
    kb, vb = _bits(kd), _bits(vd)
    for bits, vals in ((kb, kd), (vb, vd)):
        back = torch.from_numpy(bits.astype(np.int32) << 16).view(torch.float32).double().numpy()
        assert np.array_equal(back, vals)
    o8, l8 = oracle.paged_decode_fp8(q, k8, v8, ks, vs, bt, sl, c.scale)
    ob, lb = oracle.paged_decode(q, kb, vb, bt, sl, c.scale)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_fp8_decode_hand_placed_scales():
    # one sequence of 3 keys over pages [1, 0] (P = 2), one head, D = 4, scale 1.
    # K codes are one-hot 1.0 in dim 0 and q = e0, so the scores are the key scales.
    # V codes are one-hot 1.0 in dim j for key j, so out[j] = w_j * v_scale_j.
    P, D = 2, 4
    k8 = np.zeros((2, P, 1, D), np.uint8)
    v8 = np.zeros((2, P, 1, D), np.uint8)
    ks = np.full((2, 1, P), np.nan, np.float32)  # slot (page 0, slot 1) is never read
    vs = np.full((2, 1, P), np.nan, np.float32)
    keys = [(1, 0, 1.0, 4.0), (1, 1, 2.0, 8.0), (0, 0, 0.5, 16.0)]  # (page, slot, k scale, v scale)
    for j, (pg, slot, ksc, vsc) in enumerate(keys):
        k8[pg, slot, 0, 0] = 0x38
        v8[pg, slot, 0, j] = 0x38
        ks[pg, 0, slot] = ksc
        vs[pg, 0, slot] = vsc
    k8[0, 1, 0, :] = 0x7F  # NaN codes in the unused slot
    q = _bits(np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32))
    out, lse = oracle.paged_decode_fp8(q, k8, v8, ks, vs, np.array([[1, 0]], np.int32), np.array([3], np.int32), 1.0)
    z = math.exp(1.0) + math.exp(2.0) + math.exp(0.5)
    want = [math.exp(1.0) / z * 4.0, math.exp(2.0) / z * 8.0, math.exp(0.5) / z * 16.0, 0.0]
    assert np.allclose(out[0, 0], want, rtol=1e-14, atol=0)
    assert lse[0, 0] == pytest.approx(math.log(z), rel=1e-15)


# ------------------------------------------------------------------ quantise-and-append

def test_kv_append_fp8_hand_case():
    P, Hkv, D = 4, 2, 64
    k8 = np.full((3, P, Hkv, D), 0x55, np.uint8)
    v8 = k8.copy()
    ks = np.full((3, Hkv, P), 7.0, np.float32)
    vs = ks.copy()
    bt = np.array([[2, 0], [1, 2]], np.int32)
    kn = np.zeros((2, Hkv, D), np.float32)
    kn[0, 1, 0] = 3.0     # sequence 0, head 1: scale 2^-7, code of 3 * 2^7 = 384
    kn[1, 0, 5] = -0.5    # sequence 1, head 0: scale 2^-9, code of -256
    vn = -kn
    pos = np.array([5, -1], np.int32)  # sequence 0 writes key 5 -> page bt[0][1] = 0, slot 1; sequence 1 skips
    rk, rv, rks, rvs, rej = oracle.kv_append_fp8(_bits(kn), _bits(vn), bt, pos, k8, v8, ks, vs)
    assert rej == 0
    assert rks[0, 1, 1] == 2.0 ** -7 and rvs[0, 1, 1] == 2.0 ** -7 and rks[0, 0, 1] == 2.0 ** -64
    assert rk[0, 1, 1, 0] == 0x7C and rv[0, 1, 1, 0] == 0xFC  # 384 = 1.5 * 2^8
    assert np.all(rk[0, 1, 1, 1:] == 0) and np.all(rk[0, 1, 0] == 0)
    changed = (rk != k8).any(axis=(2, 3))
    assert changed.sum() == 1 and changed[0, 1]
    # rejected: a position past the table and a bad page id leave the pools untouched
    for bad_pos, bad_bt in (([8, -1], bt), ([1, -1], np.array([[5, 0], [1, 2]], np.int32))):
        r = oracle.kv_append_fp8(_bits(kn), _bits(vn), bad_bt, np.array(bad_pos, np.int32), k8, v8, ks, vs)
        assert r[4] == 1 and np.array_equal(r[0], k8) and np.array_equal(r[2], ks)
