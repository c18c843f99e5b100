"""ctypes harness around the float64 C oracle (nvfp4_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check of the
build entry point and the CPU-baseline leg of the benchmark; never by the
library.  It shares no code with the CUDA path; it receives the same seeded
inputs (numpy / CPU torch arrays) and its own host copies of the cache.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_HDR = os.path.join(_HERE, "nvfp4_oracle.h")
_SO = os.path.join(_HERE, "_build", "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no fast-math).

    NVFP4_ORACLE_SO overrides the library path (used by the mutation test,
    which loads deliberately broken copies of the oracle)."""
    if os.environ.get("NVFP4_ORACLE_SO"):
        return os.environ["NVFP4_ORACLE_SO"]
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               "-Wall", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class OrcCache(C.Structure):
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


class OrcPageTable(C.Structure):
    _fields_ = [("kv_indices", C.c_void_p), ("kv_indptr", C.c_void_p),
                ("last_page_len", C.c_void_p), ("batch", C.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_e2m1_value.restype = C.c_double
            L.orc_e2m1_value.argtypes = [C.c_uint8]
            L.orc_e4m3_value.restype = C.c_double
            L.orc_e4m3_value.argtypes = [C.c_uint8]
            L.orc_e2m1_encode.restype = C.c_uint8
            L.orc_e2m1_encode.argtypes = [C.c_double]
            L.orc_e4m3_encode.restype = C.c_uint8
            L.orc_e4m3_encode.argtypes = [C.c_double]
            L.orc_bf16_value.restype = C.c_double
            L.orc_bf16_value.argtypes = [C.c_uint16]
            L.orc_quantize_block16.restype = None
            L.orc_quantize_block16.argtypes = [C.c_void_p, C.c_double,
                                               C.c_void_p, C.c_void_p]
            L.orc_kv_len.restype = C.c_int64
            L.orc_kv_len.argtypes = [C.POINTER(OrcPageTable), C.c_int32, C.c_int32]
            L.orc_quantize_append.restype = C.c_int
            L.orc_quantize_append.argtypes = [
                C.POINTER(OrcCache), C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                C.c_int64, C.c_int64, C.c_int32, C.c_void_p, C.c_void_p,
                C.POINTER(OrcPageTable)]
            L.orc_dequant_row.restype = None
            L.orc_dequant_row.argtypes = [C.POINTER(OrcCache), C.c_int, C.c_int32,
                                          C.c_int32, C.c_int32, C.c_void_p]
            L.orc_attention_unit.restype = C.c_int
            L.orc_attention_unit.argtypes = [
                C.POINTER(OrcCache), C.POINTER(OrcPageTable), C.c_void_p,
                C.c_void_p, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                C.c_double, C.c_int32, C.c_int32, C.c_int64, C.c_void_p,
                C.c_void_p]
            L.orc_attention_unit_fp4qp.restype = C.c_int
            L.orc_attention_unit_fp4qp.argtypes = [
                C.POINTER(OrcCache), C.POINTER(OrcPageTable), C.c_void_p,
                C.c_void_p, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                C.c_double, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
            L.orc_merge_states.restype = None
            L.orc_merge_states.argtypes = [C.c_int32, C.c_int32, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_void_p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _np(t):
    """CPU torch tensor (or numpy array) -> contiguous numpy; bf16 -> uint16."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            a = t.numpy()
            return a.view(np.uint16) if a.dtype == np.int16 else a
    except ImportError:
        pass
    return np.ascontiguousarray(t)


# ---- scalars -------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(b: int) -> float:
    return lib().orc_e4m3_value(b)


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(x)


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(x)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def quantize_block16(x, g: float):
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    assert x.shape == (16,)
    packed = np.zeros(8, np.uint8)
    sf = np.zeros(1, np.uint8)
    lib().orc_quantize_block16(_ptr(x), g, _ptr(packed), _ptr(sf))
    return packed, int(sf[0])


def merge_states(o_partial, lse_partial):
    o = np.ascontiguousarray(np.asarray(o_partial, np.float64))
    l = np.ascontiguousarray(np.asarray(lse_partial, np.float64))
    n, d = o.shape
    out = np.zeros(d, np.float64)
    lse = np.zeros(1, np.float64)
    lib().orc_merge_states(n, d, _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    return out, float(lse[0])


# ---- paged cache ---------------------------------------------------------

class Cache:
    """Host buffers of a paged NVFP4 cache laid out by a ``CacheLayout``."""

    def __init__(self, layout, k_global_scale: float, v_global_scale: float,
                 fill: int = 0):
        self.layout = layout
        self.k_global_scale = float(k_global_scale)
        self.v_global_scale = float(v_global_scale)
        self.bufs = {w: np.full(layout.nbytes(w), fill, np.uint8)
                     for w in ("k_data", "v_data", "k_sf", "v_sf")}
        self._s = OrcCache()
        rows = layout.rows()
        for w, pre in (("k_data", "k"), ("v_data", "v"), ("k_sf", "k_sf"),
                       ("v_sf", "v_sf")):
            setattr(self._s, w, self.bufs[w].ctypes.data)
            sp, ss, sh = layout.strides(rows[w])
            setattr(self._s, pre + "_stride_page", sp)
            setattr(self._s, pre + "_stride_slot", ss)
            setattr(self._s, pre + "_stride_head", sh)
        self._s.num_pages = layout.num_pages
        self._s.page_size = layout.page_size
        self._s.num_kv_heads = layout.num_kv_heads
        self._s.head_dim_qk = layout.head_dim_qk
        self._s.head_dim_vo = layout.head_dim_vo
        self._s.k_global_scale = self.k_global_scale
        self._s.v_global_scale = self.v_global_scale

    @property
    def struct(self):
        return C.byref(self._s)


class PageTable:
    def __init__(self, kv_indices, kv_indptr, last_page_len):
        self.kv_indices = _np(kv_indices).astype(np.int32)
        self.kv_indptr = _np(kv_indptr).astype(np.int32)
        self.last_page_len = _np(last_page_len).astype(np.int32)
        self._s = OrcPageTable(self.kv_indices.ctypes.data,
                               self.kv_indptr.ctypes.data,
                               self.last_page_len.ctypes.data,
                               len(self.kv_indptr) - 1)

    @classmethod
    def of(cls, batch):
        return cls(batch.kv_indices, batch.kv_indptr, batch.last_page_len)

    @property
    def struct(self):
        return C.byref(self._s)


def quantize_append(cache: Cache, pt: PageTable, tokens) -> int:
    """Quantise a TokenSet (bf16 K [n,H,Dk], V [n,H,Dv]) into the cache."""
    k = _np(tokens.k)
    v = _np(tokens.v)
    bi = _np(tokens.batch_idx).astype(np.int32)
    pos = _np(tokens.positions).astype(np.int32)
    n = k.shape[0]
    if n == 0:
        return 0
    return lib().orc_quantize_append(
        cache.struct, _ptr(k), k.shape[1] * k.shape[2], k.shape[2], _ptr(v),
        v.shape[1] * v.shape[2], v.shape[2], n, _ptr(bi), _ptr(pos), pt.struct)


def dequant_row(cache: Cache, which: int, page: int, slot: int, head: int):
    dim = cache.layout.head_dim_qk if which == 0 else cache.layout.head_dim_vo
    out = np.zeros(dim, np.float64)
    lib().orc_dequant_row(cache.struct, which, page, slot, head, _ptr(out))
    return out


def attention(cache: Cache, pt: PageTable, qo_indptr, q, num_qo_heads: int,
              causal: bool, sm_scale: float, units=None, chunk_tokens: int = 0,
              out=None, lse=None):
    """Exact attention; ``units`` = iterable of (request, kv_head) to compute
    (default all).  Returns fp64 out [rows, Hq, Dv] and lse [rows, Hq]; rows
    not computed stay NaN."""
    qo = _np(qo_indptr).astype(np.int32)
    qb = _np(q)
    rows = int(qo[-1])
    Hkv = cache.layout.num_kv_heads
    if out is None:
        out = np.full((rows, num_qo_heads, cache.layout.head_dim_vo), np.nan)
    if lse is None:
        lse = np.full((rows, num_qo_heads), np.nan)
    if units is None:
        units = [(b, h) for b in range(len(qo) - 1) for h in range(Hkv)]
    L = lib()
    for b, h in units:
        rc = L.orc_attention_unit(cache.struct, pt.struct, _ptr(qo), _ptr(qb),
                                  qb.shape[1] * qb.shape[2], qb.shape[2],
                                  num_qo_heads, int(causal), sm_scale, b, h,
                                  chunk_tokens, _ptr(out), _ptr(lse))
        if rc != 0:
            raise RuntimeError("oracle attention failed (%d) for unit %r" % (rc, (b, h)))
    return out, lse


def attention_fp4qp(cache: Cache, pt: PageTable, qo_indptr, q, num_qo_heads: int,
                    causal: bool, sm_scale: float, units=None, out=None, lse=None):
    """Attention with the query and the probabilities quantised to FP4
    (orc_attention_unit_fp4qp); arguments and results as ``attention``."""
    qo = _np(qo_indptr).astype(np.int32)
    qb = _np(q)
    rows = int(qo[-1])
    Hkv = cache.layout.num_kv_heads
    if out is None:
        out = np.full((rows, num_qo_heads, cache.layout.head_dim_vo), np.nan)
    if lse is None:
        lse = np.full((rows, num_qo_heads), np.nan)
    if units is None:
        units = [(b, h) for b in range(len(qo) - 1) for h in range(Hkv)]
    L = lib()
    for b, h in units:
        rc = L.orc_attention_unit_fp4qp(cache.struct, pt.struct, _ptr(qo), _ptr(qb),
                                        qb.shape[1] * qb.shape[2], qb.shape[2],
                                        num_qo_heads, int(causal), sm_scale, b, h,
                                        _ptr(out), _ptr(lse))
        if rc != 0:
            raise RuntimeError("oracle fp4 q/p attention failed (%d) for unit %r" % (rc, (b, h)))
    return out, lse


def cache_from_batch(batch, layout: str = "HND", fill: int = 0,
                     pad_page_bytes: int = 0, include_new: bool = True):
    """Oracle-quantised cache holding a Batch's prefix (and new) tokens."""
    c = Cache(batch.cache_layout(layout, pad_page_bytes), batch.k_global_scale,
              batch.v_global_scale, fill)
    pt = PageTable.of(batch)
    rc = quantize_append(c, pt, batch.prefix)
    if rc == 0 and include_new:
        rc = quantize_append(c, pt, batch.new)
    if rc != 0:
        raise RuntimeError("oracle quantize_append failed (%d)" % rc)
    return c, pt
