"""ctypes declarations of the C ABI in include/nvfp4kv.h.

The library must be built (``build.build()``); there is no fallback: a
missing or stale library raises instead of computing anything elsewhere.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID_ARGUMENT = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE_TOO_SMALL = 3
ERR_CUDA = 4
ERR_DEVICE_CHECK = 5
ERR_PLAN_MISMATCH = 6
FLAG_BAD_PAGE_INDEX = 0x1
FLAG_BAD_APPEND_TARGET = 0x2
FLAG_COPY_TIMEOUT = 0x4
FLAG_BAD_LIVE_LENGTH = 0x8
FLAG_PACE_TIMEOUT = 0x10


class PagedCacheStruct(C.Structure):
    _fields_ = [("k_data", C.c_void_p), ("v_data", C.c_void_p),
                ("k_sf", C.c_void_p), ("v_sf", C.c_void_p)] + [
        (n, C.c_int64) for n in (
            "k_stride_page", "k_stride_slot", "k_stride_head",
            "v_stride_page", "v_stride_slot", "v_stride_head",
            "k_sf_stride_page", "k_sf_stride_slot", "k_sf_stride_head",
            "v_sf_stride_page", "v_sf_stride_slot", "v_sf_stride_head")] + [
        (n, C.c_int32) for n in ("num_pages", "page_size", "num_kv_heads",
                                 "head_dim_qk", "head_dim_vo")] + [
        ("k_global_scale", C.c_float), ("v_global_scale", C.c_float)]


class PlanOptions(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "causal", "disable_split", "max_splits", "force_chunk_tokens", "kernel",
        "num_sms", "ctas_per_sm", "out_dtype")] + [("device_last_page_len", C.c_void_p)]


class PlanInfo(C.Structure):
    _fields_ = [("magic", C.c_uint32)] + [(n, C.c_int32) for n in (
        "batch", "num_qo_heads", "num_kv_heads", "head_dim_qk", "head_dim_vo",
        "page_size", "causal", "kernel", "num_units", "row_blocks",
        "rows_per_block", "warps", "split", "chunk_pages",
        "max_units_per_request", "total_qo_rows", "num_sms", "ctas_per_sm",
        "smem_bytes", "device", "out_dtype")] + [
        ("num_partials", C.c_int64), ("total_kv_pages", C.c_int64)] + [
        (n, C.c_uint64) for n in (
            "workspace_bytes", "plan_host_bytes", "off_flags", "off_units",
            "off_merge_indptr", "off_partial_lse", "off_partial_o", "off_counters")] + [
        ("device_last_page_len", C.c_void_p), ("off_row_max", C.c_uint64)]


_vp, _i32, _i64, _u64, _f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_float
SIGNATURES = {
    "nvfp4kv_status_string": (C.c_char_p, [C.c_int]),
    "nvfp4kv_last_error_detail": (C.c_char_p, []),
    "nvfp4kv_quantize_append": (C.c_int, [
        C.POINTER(PagedCacheStruct), _vp, _i64, _i64, _vp, _i64, _i64, _i32, _vp, _vp,
        _vp, _vp, _vp, _i32, _vp, _vp]),
    "nvfp4kv_dequantize_paged": (C.c_int, [
        C.POINTER(PagedCacheStruct), _vp, _i32, _vp, _vp, _vp, _vp]),
    "nvfp4kv_decode_plan": (C.c_int, [
        _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, C.POINTER(PlanOptions), _i32,
        _vp, _u64, _vp, _u64, _vp, C.POINTER(PlanInfo)]),
    "nvfp4kv_decode_run": (C.c_int, [
        C.POINTER(PlanInfo), _vp, _i64, _i64, C.POINTER(PagedCacheStruct), _vp, _f32,
        _vp, _u64, _vp, _vp, _vp]),
    "nvfp4kv_decode_attend": (C.c_int, [
        C.POINTER(PlanInfo), _vp, _i64, _i64, C.POINTER(PagedCacheStruct), _vp, _f32,
        _vp, _u64, _vp, _vp, _vp]),
    "nvfp4kv_decode_merge": (C.c_int, [C.POINTER(PlanInfo), _vp, _u64, _vp, _vp, _vp]),
    "nvfp4kv_decode_append_run": (C.c_int, [
        C.POINTER(PlanInfo), _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
        C.POINTER(PagedCacheStruct), _vp, _f32, _vp, _u64, _vp, _vp, _vp]),
    "nvfp4kv_merge_states": (C.c_int, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
    "nvfp4kv_workspace_flags": (C.c_int, [C.POINTER(PlanInfo), _vp, C.POINTER(C.c_uint32),
                                          _i32, _vp]),
    "nvfp4kv_static_workspace_flags": (C.c_int, [C.POINTER(PlanInfo),
                                                 C.POINTER(C.c_uint32), _i32, _vp]),
    "nvfp4kv_decode_run_static": (C.c_int, [
        C.POINTER(PlanInfo), _vp, _vp, _i64, _i64, C.POINTER(PagedCacheStruct), _vp, _f32,
        _vp, _vp, _vp]),
}


def header_functions(path=None):
    """Names of the functions include/nvfp4kv.h declares."""
    path = path or os.path.join(_build.INCLUDE, "nvfp4kv.h")
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(nvfp4kv_\w+)\s*\(",
                                 text, flags=re.M)))


def load(build_if_missing: bool = True):
    """Load libnvfp4kv.so (building it in-tree first when asked)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise ImportError("libnvfp4kv.so is not built (%s); run "
                                  "__graft_entry__.build()" % path)
            lib = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class NvFp4KvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__("%s failed: %s (%s)" % (where, _status_name(status), detail))
        self.status = status
        self.detail = detail


def _status_name(st):
    return load().nvfp4kv_status_string(st).decode()


def check(status: int, where: str):
    if status != OK:
        raise NvFp4KvError(status, where, load().nvfp4kv_last_error_detail().decode())
    return status
