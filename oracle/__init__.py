"""CPU fp64 oracle for paged GQA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product library never touches it,
and it imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, double precision), compiled with
gcc into ``oracle/_build/liboracle.so`` on first use.  This module only marshals
numpy arrays into that library.

Functions: ``paged_decode`` (decode attention by the definition), ``merge`` (the
log-sum-exp combine of split partials), ``kv_append`` (the paged cache write).

Pins (see ``tests/test_oracle.py``): single-token rows, constant V, all-equal K,
hand-derived golden cases, physical-page and page-size invariance, a brute-force
comparison with torch's float64 scaled-dot-product attention, merge
associativity, scale -> 0, the GQA head mapping, and poisoned padding.
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
    if select is None:
        sel = None
        out = np.empty((B, Hq, D), np.float64)
        lse = np.empty((B, Hq), np.float64)
        nsel = 0
    else:
        pairs = np.asarray(list(select), dtype=np.int64).reshape(-1, 2)
        sel = np.ascontiguousarray(pairs[:, 0] * Hq + pairs[:, 1], dtype=np.int32)
        nsel = sel.shape[0]
        out = np.empty((nsel, D), np.float64)
        lse = np.empty((nsel,), np.float64)
    rc = lib.oracle_paged_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                                 B, Hq, Hkv, D, P, num_pages, max_pages, float(scale),
                                 _ptr(sel) if sel is not None else None, nsel,
                                 _ptr(out), _ptr(lse), int(nthreads))
    if rc == 1:
        raise ValueError("a used block_table entry is outside [0, num_pages)")
    if rc != 0:
        raise ValueError("oracle_paged_decode rejected its arguments (rc=%d)" % rc)
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
