"""Paged GQA decode attention for GB300 (sm_103a): Python binding of the C library.

Every function here only marshals arguments (device pointers, sizes, the
current CUDA stream) into the C entry points of ``include/pkv.h`` with the same
names; all of the work runs in the library's CUDA kernels.  There is no
fallback: if the compiled library is missing, every call raises.

Build the library with ``python -m paged_kv_gqa_gb300._build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PkvError", "load", "status_string", "plan_query", "paged_decode_attn_workspace_size",
    "paged_decode_attn", "paged_decode_attn_ex", "split_kv_merge", "pkv_check_status",
    "pkv_reset_status", "pkv_selftest_wait_timeout", "paged_decode_attn_static_scratch", "paged_kv_append",
    "paged_decode_attn_fp8", "paged_kv_append_fp8", "quantize_pool_fp8", "paged_prefill_attn",
    "paged_prefill_attn_workspace_size", "prefill_plan_query", "set_programmatic_launch", "set_prefill_tensor_cores",
    "set_cluster_merge", "EXPORTED_SYMBOLS",
    "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

STATUS = {
    0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED", -3: "PKV_ERR_MISALIGNED",
    -4: "PKV_ERR_WORKSPACE_TOO_SMALL", -5: "PKV_ERR_CUDA", -6: "PKV_ERR_BAD_PAGE_INDEX",
    -7: "PKV_ERR_DEVICE_TIMEOUT", -8: "PKV_ERR_BAD_SEQ_LEN", -9: "PKV_ERR_BAD_QO_INDPTR",
}

# Every symbol include/pkv.h declares.
EXPORTED_SYMBOLS = [
    "pkv_status_string", "pkv_version", "pkv_plan_query", "paged_decode_attn_workspace_size",
    "paged_decode_attn_workspace_size_ex", "paged_decode_attn", "paged_decode_attn_ex", "split_kv_merge",
    "pkv_check_status", "pkv_reset_status", "pkv_selftest_wait_timeout", "paged_decode_attn_static_scratch",
    "paged_kv_append", "paged_decode_attn_fp8", "paged_kv_append_fp8", "pkv_plan_query_kv",
    "paged_decode_attn_workspace_size_kv", "paged_prefill_attn", "paged_prefill_attn_fp8",
    "pkv_plan_query_prefill", "paged_prefill_attn_workspace_size", "pkv_set_programmatic_launch",
    "pkv_set_prefill_tensor_cores", "pkv_set_cluster_merge", "pkv_set_adaptive_splits",
]

KV_DTYPES = {"bf16": 0, "fp8": 1}


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s (%d)" % (where, STATUS.get(status, "unknown"), status))


class PkvPlan(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int), ("chunk_tokens", ctypes.c_int), ("stage_tokens", ctypes.c_int),
                ("warps", ctypes.c_int), ("ring_stages", ctypes.c_int), ("blocks_per_sm", ctypes.c_int),
                ("grid_blocks", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("merge_needed", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("q_tiles", ctypes.c_int), ("rows_per_block", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Loads the compiled library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("paged_kv_gqa_gb300: CUDA library %s is missing; build it with "
                               "`python -m paged_kv_gqa_gb300._build`" % path)
        lib = ctypes.CDLL(path)
        P, I, F, S, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint
        sig = {
            "pkv_status_string": (ctypes.c_char_p, [I]),
            "pkv_version": (I, []),
            "pkv_plan_query": (I, [I, I, I, I, I, I, I, I, ctypes.POINTER(PkvPlan)]),
            "paged_decode_attn_workspace_size": (I, [I, I, I, I, I, I, I, ctypes.POINTER(S)]),
            "paged_decode_attn_workspace_size_ex": (I, [I, I, I, I, I, I, I, I, ctypes.POINTER(S)]),
            "paged_decode_attn": (I, [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, S, P]),
            "paged_decode_attn_ex": (I, [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, S, I, P]),
            "split_kv_merge": (I, [P, P, I, I, I, I, P, P, P]),
            "pkv_check_status": (I, [P, P, ctypes.POINTER(I)]),
            "pkv_reset_status": (I, [P, P]),
            "pkv_selftest_wait_timeout": (I, [P, U, P]),
            "paged_decode_attn_static_scratch": (I, [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P]),
            "paged_kv_append": (I, [P, P, P, P, I, I, I, I, I, I, P, P, P, P]),
            "paged_decode_attn_fp8": (I, [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, S, I, P]),
            "pkv_plan_query_kv": (I, [I, I, I, I, I, I, I, I, I, ctypes.POINTER(PkvPlan)]),
            "paged_decode_attn_workspace_size_kv": (I, [I, I, I, I, I, I, I, I, I, ctypes.POINTER(S)]),
            "paged_prefill_attn": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, P, P, P, S, I, P]),
            "paged_prefill_attn_fp8": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, P, P, P, S, I,
                                           P]),
            "pkv_plan_query_prefill": (I, [I, I, I, I, I, I, I, I, I, I, I, ctypes.POINTER(PkvPlan)]),
            "pkv_set_programmatic_launch": (I, [I]),
            "pkv_set_cluster_merge": (I, [I]),
            "pkv_set_adaptive_splits": (I, [I]),
            "pkv_set_prefill_tensor_cores": (I, [I]),
            "paged_prefill_attn_workspace_size": (I, [I, I, I, I, I, I, I, I, I, I, I, ctypes.POINTER(S)]),
            "paged_kv_append_fp8": (I, [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise PkvError(status, where)


def set_programmatic_launch(enable: bool) -> bool:
    """Turns programmatic dependent launch on or off for every later launch; returns the old setting."""
    return bool(load().pkv_set_programmatic_launch(int(bool(enable))))


def set_cluster_merge(enable: bool) -> bool:
    """Decode calls with 2-8 splits merge them inside a thread-block cluster (on, the default)
    or through the workspace (off); returns the old setting."""
    return bool(load().pkv_set_cluster_merge(int(bool(enable))))


def set_adaptive_splits(enable: bool) -> bool:
    """Decode calls with the automatic split count size their splits on the device from the
    batch's actual lengths (on) or from the block table's width (off, the default); returns
    the old setting."""
    return bool(load().pkv_set_adaptive_splits(int(bool(enable))))


TC_MODES = {"off": 0, "auto": 1, "always": 2, "rows128": 3}


def set_prefill_tensor_cores(mode="auto") -> str:
    """Routing of multi-row calls with more than 32 rows per group (D=128, scale > 0; a
    group of at most 32 rows always takes the mma.sync kernel): "off" = the mma.sync kernel;
    "auto" (default) = groups of 33-127 rows on the tcgen05 kernel with 128 rows per CTA when
    the block table spans >= 8192 keys, else the mma.sync kernel; larger groups on the tcgen05
    kernel with 256 rows per CTA when the group has them and that grid (key splits included)
    has a CTA per two SMs, else with 128 rows; "always" = the tcgen05 kernel (256 rows per CTA
    where the group has them); "rows128" = the tcgen05 kernel with 128 rows per CTA.  The fp8
    cache takes the 128-row kernel wherever a mode names the tcgen05 kernel.  True/False mean
    "auto"/"off".  Returns the previous mode."""
    if isinstance(mode, bool):
        mode = "auto" if mode else "off"
    if mode not in TC_MODES:
        raise ValueError("mode must be one of %s" % sorted(TC_MODES))
    old = load().pkv_set_prefill_tensor_cores(TC_MODES[mode])
    if old < 0:
        raise PkvError(old, "pkv_set_prefill_tensor_cores")
    return {v: k for k, v in TC_MODES.items()}[old]


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def plan_query(B, Hq, Hkv, D, page_size, max_pages, num_sms, num_splits=0, cache="bf16") -> dict:
    plan = PkvPlan()
    _check(load().pkv_plan_query_kv(B, Hq, Hkv, D, page_size, max_pages, num_sms, num_splits, KV_DTYPES[cache],
                                    ctypes.byref(plan)), "pkv_plan_query_kv")
    return plan.as_dict()


# ----------------------------------------------------------------- tensor helpers (torch only for plumbing)

def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev_ptr(t, dtype, name, ndim=None):
    torch = _torch()
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dimensions, got shape %s" % (name, ndim, tuple(t.shape)))
    return ctypes.c_void_p(t.data_ptr())


def paged_decode_attn_workspace_size(B, Hq, Hkv, D, page_size, max_pages, device=None, num_splits=0,
                                     cache="bf16") -> int:
    torch = _torch()
    dev = torch.cuda.current_device() if device is None else int(device)
    n = ctypes.c_size_t(0)
    _check(load().paged_decode_attn_workspace_size_kv(B, Hq, Hkv, D, page_size, max_pages, dev, num_splits,
                                                      KV_DTYPES[cache], ctypes.byref(n)),
           "paged_decode_attn_workspace_size_kv")
    return n.value


def paged_decode_attn_ex(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, workspace,
                         num_splits=0, stream=None):
    """Calls paged_decode_attn_ex on torch CUDA tensors (shapes as in include/pkv.h)."""
    torch = _torch()
    B, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q/k_cache/v_cache shapes disagree")
    if tuple(out.shape) != (B, Hq, D):
        raise ValueError("out must be [B, Hq, D]")
    if lse is not None and tuple(lse.shape) != (B, Hq):
        raise ValueError("lse must be [B, Hq]")
    max_pages = block_table.shape[1]
    st = load().paged_decode_attn_ex(
        _dev_ptr(q, torch.bfloat16, "q", 3), _dev_ptr(k_cache, torch.bfloat16, "k_cache", 4),
        _dev_ptr(v_cache, torch.bfloat16, "v_cache", 4), _dev_ptr(block_table, torch.int32, "block_table", 2),
        _dev_ptr(seq_lens, torch.int32, "seq_lens", 1), B, Hq, Hkv, D, P, num_pages, max_pages,
        ctypes.c_float(scale), _dev_ptr(out, torch.bfloat16, "out", 3),
        _dev_ptr(lse, torch.float32, "lse", 2) if lse is not None else None,
        _dev_ptr(workspace, workspace.dtype, "workspace"), workspace.numel() * workspace.element_size(),
        int(num_splits), _stream_handle(stream))
    _check(st, "paged_decode_attn_ex")
    return out, lse


def paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, workspace, stream=None):
    """Calls paged_decode_attn (automatic split count) on torch CUDA tensors."""
    return paged_decode_attn_ex(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, workspace,
                                num_splits=0, stream=stream)


def split_kv_merge(partial_out, partial_lse, out, lse=None, stream=None):
    """Calls split_kv_merge: partial_out [S,B,Hq,D] f32, partial_lse [S,B,Hq] f32 -> out bf16, lse f32."""
    torch = _torch()
    S, B, Hq, D = partial_out.shape
    if tuple(partial_lse.shape) != (S, B, Hq):
        raise ValueError("partial_lse must be [S, B, Hq]")
    st = load().split_kv_merge(_dev_ptr(partial_out, torch.float32, "partial_out", 4),
                               _dev_ptr(partial_lse, torch.float32, "partial_lse", 3), S, B, Hq, D,
                               _dev_ptr(out, torch.bfloat16, "out", 3),
                               _dev_ptr(lse, torch.float32, "lse", 2) if lse is not None else None,
                               _stream_handle(stream))
    _check(st, "split_kv_merge")
    return out, lse


def pkv_check_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the workspace's device status word."""
    v = ctypes.c_int(0)
    _check(load().pkv_check_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(stream), ctypes.byref(v)),
           "pkv_check_status")
    return v.value


def pkv_reset_status(workspace, stream=None):
    _check(load().pkv_reset_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(stream)),
           "pkv_reset_status")


def pkv_selftest_wait_timeout(workspace, timeout_us=1000, stream=None):
    _check(load().pkv_selftest_wait_timeout(ctypes.c_void_p(workspace.data_ptr()), int(timeout_us),
                                            _stream_handle(stream)), "pkv_selftest_wait_timeout")


def paged_decode_attn_static_scratch(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse,
                                     device_status=None, stream=None):
    """Calls paged_decode_attn_static_scratch: decode without a caller workspace, for
    callers that cannot allocate device memory (the library's fixed scratch is used)."""
    torch = _torch()
    B, Hq, D = q.shape
    num_pages, P, Hkv, _ = k_cache.shape
    st = load().paged_decode_attn_static_scratch(
        _dev_ptr(q, torch.bfloat16, "q", 3), _dev_ptr(k_cache, torch.bfloat16, "k_cache", 4),
        _dev_ptr(v_cache, torch.bfloat16, "v_cache", 4), _dev_ptr(block_table, torch.int32, "block_table", 2),
        _dev_ptr(seq_lens, torch.int32, "seq_lens", 1), B, Hq, Hkv, D, P, num_pages, block_table.shape[1],
        ctypes.c_float(scale), _dev_ptr(out, torch.bfloat16, "out", 3),
        _dev_ptr(lse, torch.float32, "lse", 2) if lse is not None else None,
        _dev_ptr(device_status, torch.int32, "device_status") if device_status is not None else None,
        _stream_handle(stream))
    _check(st, "paged_decode_attn_static_scratch")
    return out, lse


def paged_kv_append(k_new, v_new, block_table, positions, k_cache, v_cache, status=None, stream=None):
    """Calls paged_kv_append: writes k_new/v_new [B, Hkv, D] into the page pools at positions[b]."""
    torch = _torch()
    B, Hkv, D = k_new.shape
    num_pages, P, Hkv2, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or tuple(v_new.shape) != tuple(k_new.shape) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_new/v_new/k_cache/v_cache shapes disagree")
    st = load().paged_kv_append(
        _dev_ptr(k_new, torch.bfloat16, "k_new", 3), _dev_ptr(v_new, torch.bfloat16, "v_new", 3),
        _dev_ptr(block_table, torch.int32, "block_table", 2), _dev_ptr(positions, torch.int32, "positions", 1),
        B, Hkv, D, P, num_pages, block_table.shape[1], _dev_ptr(k_cache, torch.bfloat16, "k_cache", 4),
        _dev_ptr(v_cache, torch.bfloat16, "v_cache", 4),
        ctypes.c_void_p(status.data_ptr()) if status is not None else None, _stream_handle(stream))
    _check(st, "paged_kv_append")


# ----------------------------------------------------------------- fp8 (e4m3) cache

def paged_decode_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, scale, out, lse, workspace,
                          num_splits=0, stream=None):
    """Calls paged_decode_attn_fp8: k_cache/v_cache uint8 e4m3 codes [num_pages, P, Hkv, D],
    k_scale/v_scale float32 [num_pages, Hkv, P]; the rest as for paged_decode_attn_ex."""
    torch = _torch()
    B, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q/k_cache/v_cache shapes disagree")
    if tuple(k_scale.shape) != (num_pages, Hkv, P) or tuple(v_scale.shape) != (num_pages, Hkv, P):
        raise ValueError("k_scale/v_scale must be [num_pages, Hkv, page_size]")
    if tuple(out.shape) != (B, Hq, D):
        raise ValueError("out must be [B, Hq, D]")
    if lse is not None and tuple(lse.shape) != (B, Hq):
        raise ValueError("lse must be [B, Hq]")
    st = load().paged_decode_attn_fp8(
        _dev_ptr(q, torch.bfloat16, "q", 3), _dev_ptr(k_cache, torch.uint8, "k_cache", 4),
        _dev_ptr(v_cache, torch.uint8, "v_cache", 4), _dev_ptr(k_scale, torch.float32, "k_scale", 3),
        _dev_ptr(v_scale, torch.float32, "v_scale", 3), _dev_ptr(block_table, torch.int32, "block_table", 2),
        _dev_ptr(seq_lens, torch.int32, "seq_lens", 1), B, Hq, Hkv, D, P, num_pages, block_table.shape[1],
        ctypes.c_float(scale), _dev_ptr(out, torch.bfloat16, "out", 3),
        _dev_ptr(lse, torch.float32, "lse", 2) if lse is not None else None,
        _dev_ptr(workspace, workspace.dtype, "workspace"), workspace.numel() * workspace.element_size(),
        int(num_splits), _stream_handle(stream))
    _check(st, "paged_decode_attn_fp8")
    return out, lse


def paged_kv_append_fp8(k_new, v_new, block_table, positions, k_cache, v_cache, k_scale, v_scale, status=None,
                        stream=None):
    """Calls paged_kv_append_fp8: quantises k_new/v_new [B, Hkv, D] (bf16) into the fp8 pools
    (uint8 [num_pages, P, Hkv, D]) and their scales (float32 [num_pages, Hkv, P]) at positions[b]."""
    torch = _torch()
    B, Hkv, D = k_new.shape
    num_pages, P, Hkv2, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or tuple(v_new.shape) != tuple(k_new.shape) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_new/v_new/k_cache/v_cache shapes disagree")
    if tuple(k_scale.shape) != (num_pages, Hkv, P) or tuple(v_scale.shape) != (num_pages, Hkv, P):
        raise ValueError("k_scale/v_scale must be [num_pages, Hkv, page_size]")
    st = load().paged_kv_append_fp8(
        _dev_ptr(k_new, torch.bfloat16, "k_new", 3), _dev_ptr(v_new, torch.bfloat16, "v_new", 3),
        _dev_ptr(block_table, torch.int32, "block_table", 2), _dev_ptr(positions, torch.int32, "positions", 1),
        B, Hkv, D, P, num_pages, block_table.shape[1], _dev_ptr(k_cache, torch.uint8, "k_cache", 4),
        _dev_ptr(v_cache, torch.uint8, "v_cache", 4), _dev_ptr(k_scale, torch.float32, "k_scale", 3),
        _dev_ptr(v_scale, torch.float32, "v_scale", 3),
        ctypes.c_void_p(status.data_ptr()) if status is not None else None, _stream_handle(stream))
    _check(st, "paged_kv_append_fp8")


def quantize_pool_fp8(k_cache, v_cache, stream=None):
    """Quantises whole bf16 pools [num_pages, P, Hkv, D] into new fp8 pools and scales with one
    paged_kv_append_fp8 launch (one row per (page, slot), a one-page table per row)."""
    torch = _torch()
    num_pages, P, Hkv, D = k_cache.shape
    dev = k_cache.device
    n = num_pages * P
    rows = torch.arange(n, device=dev, dtype=torch.int32)
    table = (rows // P).reshape(n, 1).contiguous()
    pos = (rows % P).contiguous()
    k8 = torch.empty((num_pages, P, Hkv, D), dtype=torch.uint8, device=dev)
    v8 = torch.empty_like(k8)
    ks = torch.empty((num_pages, Hkv, P), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    paged_kv_append_fp8(k_cache.reshape(n, Hkv, D), v_cache.reshape(n, Hkv, D), table, pos, k8, v8, ks, vs,
                        stream=stream)
    return k8, v8, ks, vs


# ----------------------------------------------------------------- several query rows per sequence

def prefill_plan_query(B, Hq, Hkv, D, page_size, max_pages, total_q, max_q_len, num_sms, num_splits=0,
                       cache="bf16") -> dict:
    plan = PkvPlan()
    _check(load().pkv_plan_query_prefill(B, Hq, Hkv, D, page_size, max_pages, total_q, max_q_len, num_sms,
                                         num_splits, KV_DTYPES[cache], ctypes.byref(plan)), "pkv_plan_query_prefill")
    return plan.as_dict()


def paged_prefill_attn_workspace_size(B, Hq, Hkv, D, page_size, max_pages, total_q, max_q_len, device=None,
                                      num_splits=0, cache="bf16") -> int:
    torch = _torch()
    dev = torch.cuda.current_device() if device is None else int(device)
    n = ctypes.c_size_t(0)
    _check(load().paged_prefill_attn_workspace_size(B, Hq, Hkv, D, page_size, max_pages, total_q, max_q_len, dev,
                                                    num_splits, KV_DTYPES[cache], ctypes.byref(n)),
           "paged_prefill_attn_workspace_size")
    return n.value


def paged_prefill_attn(q, k_cache, v_cache, qo_indptr, block_table, seq_lens, max_q_len, scale, out, lse, workspace,
                       causal=True, num_splits=0, stream=None, fp8_scales=None):
    """Calls paged_prefill_attn (or paged_prefill_attn_fp8 when fp8_scales = (k_scale, v_scale)):
    q/out [total_q, Hq, D], qo_indptr [B+1], the cache and table as for decode."""
    torch = _torch()
    total_q, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k_cache.shape
    B = seq_lens.shape[0]
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q/k_cache/v_cache shapes disagree")
    if tuple(out.shape) != (total_q, Hq, D) or (lse is not None and tuple(lse.shape) != (total_q, Hq)):
        raise ValueError("out must be [total_q, Hq, D] and lse [total_q, Hq]")
    if tuple(qo_indptr.shape) != (B + 1,):
        raise ValueError("qo_indptr must be [B+1]")
    common = (_dev_ptr(qo_indptr, torch.int32, "qo_indptr", 1), _dev_ptr(block_table, torch.int32, "block_table", 2),
              _dev_ptr(seq_lens, torch.int32, "seq_lens", 1), B, Hq, Hkv, D, P, num_pages, block_table.shape[1],
              total_q, int(max_q_len), int(bool(causal)), ctypes.c_float(scale),
              _dev_ptr(out, torch.bfloat16, "out", 3), _dev_ptr(lse, torch.float32, "lse", 2) if lse is not None else None,
              _dev_ptr(workspace, workspace.dtype, "workspace"), workspace.numel() * workspace.element_size(),
              int(num_splits), _stream_handle(stream))
    if fp8_scales is None:
        st = load().paged_prefill_attn(_dev_ptr(q, torch.bfloat16, "q", 3), _dev_ptr(k_cache, torch.bfloat16, "k_cache", 4),
                                       _dev_ptr(v_cache, torch.bfloat16, "v_cache", 4), *common)
    else:
        ks, vs = fp8_scales
        st = load().paged_prefill_attn_fp8(_dev_ptr(q, torch.bfloat16, "q", 3), _dev_ptr(k_cache, torch.uint8, "k_cache", 4),
                                           _dev_ptr(v_cache, torch.uint8, "v_cache", 4),
                                           _dev_ptr(ks, torch.float32, "k_scale", 3), _dev_ptr(vs, torch.float32, "v_scale", 3),
                                           *common)
    _check(st, "paged_prefill_attn")
    return out, lse