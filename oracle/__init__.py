"""CPU fp64 oracle for paged GQA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product library never touches it,
and it imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, double precision), compiled with
gcc into ``oracle/_build/liboracle.so`` on first use.  This module only marshals
numpy arrays into that library.

Functions: ``paged_decode`` (decode attention by the definition), ``paged_prefill``
(several query rows per request, ragged by ``qo_indptr``, causal or not), ``merge`` (the
log-sum-exp combine of split partials), ``kv_append`` (the paged cache write), and
the FP8 KV variant: ``e4m3_value`` / ``e4m3_encode`` (the codec), ``fp8_quantize_rows``
(power-of-two row scales), ``quantize_pool`` / ``dequantize_pool``,
``paged_decode_fp8`` and ``kv_append_fp8``.

Pins (see ``tests/test_oracle.py``): single-token rows, constant V, all-equal K,
hand-derived golden cases, physical-page and page-size invariance, a brute-force
comparison with torch's float64 scaled-dot-product attention, merge
associativity, scale -> 0, the GQA head mapping, and poisoned padding; for FP8,
code values from the format's definition, torch's float8_e4m3fn codec, rounding
ties, the quantiser's scale rule and error bound, and hand-placed scales.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (IEEE arithmetic, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
               "-pthread", "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_paged_decode.restype = i
            lib.oracle_paged_decode.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i,
                                                ctypes.c_double, p, i, p, p, i]
            lib.oracle_merge.restype = None
            lib.oracle_merge.argtypes = [p, p, i, i, i, p, p]
            lib.oracle_kv_append.restype = i
            lib.oracle_kv_append.argtypes = [p, p, p, p, i, i, i, i, i, i, p, p]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            lib.oracle_fp8_quantize_rows.restype = None
            lib.oracle_fp8_quantize_rows.argtypes = [p, i, i, p, p]
            lib.oracle_paged_decode_fp8.restype = i
            lib.oracle_paged_decode_fp8.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i,
                                                    ctypes.c_double, p, i, p, p, i]
            lib.oracle_paged_prefill.restype = i
            lib.oracle_paged_prefill.argtypes = [p, p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i,
                                                 ctypes.c_double, i, p, i, p, p, i]
            lib.oracle_kv_append_fp8.restype = i
            lib.oracle_kv_append_fp8.argtypes = [p, p, p, p, i, i, i, i, i, i, p, p, p, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_bits(x) -> np.ndarray:
    """bf16 tensors arrive as uint16 bit patterns (numpy has no bfloat16)."""
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands must be passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _select(select, B, Hq, D):
    if select is None:
        return None, 0, np.empty((B, Hq, D), np.float64), np.empty((B, Hq), np.float64)
    pairs = np.asarray(list(select), dtype=np.int64).reshape(-1, 2)
    sel = np.ascontiguousarray(pairs[:, 0] * Hq + pairs[:, 1], dtype=np.int32)
    nsel = sel.shape[0]
    return sel, nsel, np.empty((nsel, D), np.float64), np.empty((nsel,), np.float64)


def _check_rc(rc, name):
    if rc == 1:
        raise ValueError("a used block_table entry is outside [0, num_pages)")
    if rc != 0:
        raise ValueError("%s rejected its arguments (rc=%d)" % (name, rc))


def paged_decode(q_bits, k_bits, v_bits, block_table, seq_lens, scale, select=None, nthreads=0):
    """Decode attention by the plain definition, in double precision.

    q_bits   uint16 [B, Hq, D]              bf16 bit patterns
    k_bits   uint16 [num_pages, P, Hkv, D]  bf16 bit patterns
    v_bits   uint16 [num_pages, P, Hkv, D]
    block_table int32 [B, max_pages];  seq_lens int32 [B]
    scale    float (applied to q.k as given, widened to double)
    select   optional iterable of (b, h) pairs; outputs are then packed in that order
    Returns (out float64 [B, Hq, D] or [n, D], lse float64 [B, Hq] or [n]).
    """
    lib = _load()
    q = _as_bits(q_bits)
    k = _as_bits(k_bits)
    v = _as_bits(v_bits)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k.shape
    if Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    sel, nsel, out, lse = _select(select, B, Hq, D)
    rc = lib.oracle_paged_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                                 B, Hq, Hkv, D, P, num_pages, max_pages, float(scale),
                                 _ptr(sel) if sel is not None else None, nsel,
                                 _ptr(out), _ptr(lse), int(nthreads))
    _check_rc(rc, "oracle_paged_decode")
    return out, lse


def merge(partial_out, partial_lse):
    """Log-sum-exp merge of split partial states, in double precision.

    partial_out float [S, N, D] (normalised per split); partial_lse float [S, N]
    (natural log, -inf = empty split).  Returns (out [N, D], lse [N]).
    """
    lib = _load()
    po = np.ascontiguousarray(partial_out, dtype=np.float64)
    pl = np.ascontiguousarray(partial_lse, dtype=np.float64)
    S, N, D = po.shape
    if pl.shape != (S, N):
        raise ValueError("partial_lse must be [S, N]")
    out = np.empty((N, D), np.float64)
    lse = np.empty((N,), np.float64)
    lib.oracle_merge(_ptr(po), _ptr(pl), S, N, D, _ptr(out), _ptr(lse))
    return out, lse


def kv_append(k_new_bits, v_new_bits, block_table, positions, k_bits, v_bits):
    """Paged KV append on host copies: returns (k_cache, v_cache, rejected).

    k_new_bits, v_new_bits uint16 [B, Hkv, D]; positions int32 [B] (the key index to
    write; < 0 skips the sequence); k_bits, v_bits uint16 [num_pages, P, Hkv, D] are
    copied, not modified.  `rejected` counts sequences whose position or page id was
    out of range (nothing written for them).
    """
    lib = _load()
    kn = _as_bits(k_new_bits)
    vn = _as_bits(v_new_bits)
    k = np.array(_as_bits(k_bits), copy=True)
    v = np.array(_as_bits(v_bits), copy=True)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    B, Hkv, D = kn.shape
    num_pages, P, Hkv2, D2 = k.shape
    if (Hkv2, D2) != (Hkv, D) or vn.shape != kn.shape or v.shape != k.shape:
        raise ValueError("shape mismatch")
    rej = lib.oracle_kv_append(_ptr(kn), _ptr(vn), _ptr(bt), _ptr(pos), B, Hkv, D, P, num_pages, bt.shape[1],
                               _ptr(k), _ptr(v))
    return k, v, rej


# ------------------------------------------------------------------ FP8 (e4m3) KV variant

def e4m3_value(codes) -> np.ndarray:
    """Exact value (float64) of each e4m3 code (uint8 array); NaN for 0x7F / 0xFF."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.oracle_e4m3_value(i) for i in range(256)], np.float64)
    return table[c]


def e4m3_encode(values) -> np.ndarray:
    """Nearest e4m3 code of each value (ties to even, saturating at +-448)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    flat = [lib.oracle_e4m3_encode(float(x)) for x in v.reshape(-1)]
    return np.asarray(flat, dtype=np.uint8).reshape(v.shape)


def fp8_quantize_rows(x_bits, nthreads=0):
    """Quantise rows of bf16 values: x_bits uint16 [..., D] -> (codes uint8 [..., D],
    scales float32 [...]) with one power-of-two scale per row.  Rows are independent;
    large inputs are cut into contiguous row ranges quantised on parallel threads."""
    lib = _load()
    x = _as_bits(x_bits)
    D = x.shape[-1]
    N = int(np.prod(x.shape[:-1]))
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[:-1], np.float32)
    xf, cf, sf = x.reshape(N, D), codes.reshape(N, D), scales.reshape(N)
    n_th = nthreads if nthreads > 0 else (os.cpu_count() or 1)
    step = max(1 << 14, -(-N // n_th))
    ranges = [(a, min(N, a + step)) for a in range(0, N, step)]

    def run(r):
        a, b = r
        lib.oracle_fp8_quantize_rows(_ptr(xf[a:b]), b - a, D, _ptr(cf[a:b]), _ptr(sf[a:b]))

    if len(ranges) <= 1:
        for r in ranges:
            run(r)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
            list(ex.map(run, ranges))
    return codes, scales


def quantize_pool(pool_bits):
    """bf16 pool uint16 [num_pages, P, Hkv, D] -> (codes uint8 [num_pages, P, Hkv, D],
    scales float32 [num_pages, Hkv, P]): the scale layout is head-major within a page."""
    codes, scales = fp8_quantize_rows(pool_bits)
    return codes, np.ascontiguousarray(scales.transpose(0, 2, 1))


def dequantize_pool(codes, scales) -> np.ndarray:
    """codes uint8 [num_pages, P, Hkv, D], scales [num_pages, Hkv, P] -> float64 values
    code value * scale, in the pool layout."""
    vals = e4m3_value(codes)
    s = np.asarray(scales, dtype=np.float64).transpose(0, 2, 1)[..., None]
    return vals * s


def paged_decode_fp8(q_bits, k8, v8, k_scale, v_scale, block_table, seq_lens, scale, select=None, nthreads=0):
    """Decode attention over an fp8 cache: key/value elements are code value * scale.

    k8, v8 uint8 [num_pages, P, Hkv, D]; k_scale, v_scale float32 [num_pages, Hkv, P];
    the other arguments and the result are those of ``paged_decode``.
    """
    lib = _load()
    q = _as_bits(q_bits)
    k = np.ascontiguousarray(k8, dtype=np.uint8)
    v = np.ascontiguousarray(v8, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k.shape
    if Dk != D or v.shape != k.shape or ks.shape != (num_pages, Hkv, P) or vs.shape != ks.shape:
        raise ValueError("shape mismatch between q, the fp8 pools and their scales")
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    sel, nsel, out, lse = _select(select, B, Hq, D)
    rc = lib.oracle_paged_decode_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                                     B, Hq, Hkv, D, P, num_pages, max_pages, float(scale),
                                     _ptr(sel) if sel is not None else None, nsel,
                                     _ptr(out), _ptr(lse), int(nthreads))
    _check_rc(rc, "oracle_paged_decode_fp8")
    return out, lse


def kv_append_fp8(k_new_bits, v_new_bits, block_table, positions, k8, v8, k_scale, v_scale):
    """Quantise-and-append on host copies: returns (k8, v8, k_scale, v_scale, rejected).

    k_new_bits, v_new_bits uint16 [B, Hkv, D]; k8, v8 uint8 [num_pages, P, Hkv, D];
    k_scale, v_scale float32 [num_pages, Hkv, P].  Inputs are copied, not modified.
    """
    lib = _load()
    kn = _as_bits(k_new_bits)
    vn = _as_bits(v_new_bits)
    k = np.array(k8, dtype=np.uint8, copy=True)
    v = np.array(v8, dtype=np.uint8, copy=True)
    ks = np.array(k_scale, dtype=np.float32, copy=True)
    vs = np.array(v_scale, dtype=np.float32, copy=True)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    B, Hkv, D = kn.shape
    num_pages, P, Hkv2, D2 = k.shape
    if (Hkv2, D2) != (Hkv, D) or vn.shape != kn.shape or v.shape != k.shape or ks.shape != (num_pages, Hkv, P):
        raise ValueError("shape mismatch")
    rej = lib.oracle_kv_append_fp8(_ptr(kn), _ptr(vn), _ptr(bt), _ptr(pos), B, Hkv, D, P, num_pages,
                                   bt.shape[1], _ptr(k), _ptr(v), _ptr(ks), _ptr(vs))
    return k, v, ks, vs, rej


# ------------------------------------------------------------------ multi-token rows

def paged_prefill(q_bits, qo_indptr, block_table, seq_lens, scale, causal=True, k_bits=None, v_bits=None,
                  fp8=None, select=None, nthreads=0):
    """Attention for several query rows per request (ragged by qo_indptr), by the definition.

    q_bits uint16 [total_q, Hq, D]; qo_indptr int32 [B+1]; block_table int32 [B, max_pages];
    seq_lens int32 [B] (keys per request, the new tokens included).  The cache is either
    k_bits/v_bits (uint16 bf16 [num_pages, P, Hkv, D]) or fp8 = (k8, v8, k_scale, v_scale).
    causal: row i of request b (n_b rows, L_b keys) sees keys j <= L_b - n_b + i.
    select: optional (t, h) pairs.  Returns (out [total_q, Hq, D] or [n, D], lse).
    """
    lib = _load()
    q = _as_bits(q_bits)
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    total_q, Hq, D = q.shape
    B = sl.shape[0]
    if qo.shape != (B + 1,):
        raise ValueError("qo_indptr must be [B+1]")
    if fp8 is not None:
        k8, v8, ks, vs = (np.ascontiguousarray(fp8[0], dtype=np.uint8), np.ascontiguousarray(fp8[1], dtype=np.uint8),
                          np.ascontiguousarray(fp8[2], dtype=np.float32), np.ascontiguousarray(fp8[3], dtype=np.float32))
        num_pages, P, Hkv, Dk = k8.shape
        ptrs = (None, None, _ptr(k8), _ptr(v8), _ptr(ks), _ptr(vs))
    else:
        k, v = _as_bits(k_bits), _as_bits(v_bits)
        num_pages, P, Hkv, Dk = k.shape
        ptrs = (_ptr(k), _ptr(v), None, None, None, None)
    if Dk != D:
        raise ValueError("head dims of q and the cache disagree")
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    if select is None:
        sel, nsel = None, 0
        out = np.empty((total_q, Hq, D), np.float64)
        lse = np.empty((total_q, Hq), np.float64)
    else:
        pairs = np.asarray(list(select), dtype=np.int64).reshape(-1, 2)
        sel = np.ascontiguousarray(pairs[:, 0] * Hq + pairs[:, 1], dtype=np.int32)
        nsel = sel.shape[0]
        out = np.empty((nsel, D), np.float64)
        lse = np.empty((nsel,), np.float64)
    rc = lib.oracle_paged_prefill(_ptr(q), *ptrs, _ptr(qo), _ptr(bt), _ptr(sl), B, Hq, Hkv, D, P, num_pages,
                                  max_pages, total_q, float(scale), int(bool(causal)),
                                  _ptr(sel) if sel is not None else None, nsel, _ptr(out), _ptr(lse),
                                  int(nthreads))
    _check_rc(rc, "oracle_paged_prefill")
    return out, lse
