"""Python binding of the C ABI (include/nvfp4kv.h), same entry-point names.

Argument marshalling only: torch supplies device memory and the stream; every
step of the computation runs in the library's CUDA kernels.  Errors raise
``NvFp4KvError`` with the library's status and message.
"""
from __future__ import annotations

import ctypes as C
import math
from typing import Optional

import torch

from . import _lib
from ._lib import NvFp4KvError, PagedCacheStruct, PlanInfo, PlanOptions, check

__all__ = ["PagedCache", "Plan", "NvFp4KvError", "nvfp4kv_quantize_append",
           "nvfp4kv_decode_plan", "nvfp4kv_decode_run", "nvfp4kv_decode_attend",
           "nvfp4kv_decode_merge", "nvfp4kv_merge_states", "nvfp4kv_workspace_flags",
           "nvfp4kv_decode_run_static", "nvfp4kv_static_workspace_flags",
           "nvfp4kv_decode_append_run",
           "nvfp4kv_dequantize_paged"]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


class PagedCache:
    """Four caller-owned uint8 buffers of a paged NVFP4 cache plus their byte
    strides (``CacheLayout`` from workloads, or explicit tensors)."""

    def __init__(self, k_data, v_data, k_sf, v_sf, strides, num_pages,
                 num_kv_heads, head_dim_qk, head_dim_vo, k_global_scale=1.0,
                 v_global_scale=1.0, page_size=16):
        self.k_data, self.v_data, self.k_sf, self.v_sf = k_data, v_data, k_sf, v_sf
        self.strides = dict(strides)
        self.num_pages = int(num_pages)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim_qk = int(head_dim_qk)
        self.head_dim_vo = int(head_dim_vo)
        self.k_global_scale = float(k_global_scale)
        self.v_global_scale = float(v_global_scale)
        self.page_size = int(page_size)

    @classmethod
    def allocate(cls, layout, k_global_scale=1.0, v_global_scale=1.0, device="cuda",
                 fill: Optional[int] = 0):
        bufs = {}
        for w in ("k_data", "v_data", "k_sf", "v_sf"):
            n = layout.nbytes(w)
            bufs[w] = (torch.empty(n, dtype=torch.uint8, device=device) if fill is None
                       else torch.full((n,), fill, dtype=torch.uint8, device=device))
        rows = layout.rows()
        strides = {w: layout.strides(rows[w]) for w in rows}
        return cls(bufs["k_data"], bufs["v_data"], bufs["k_sf"], bufs["v_sf"], strides,
                   layout.num_pages, layout.num_kv_heads, layout.head_dim_qk,
                   layout.head_dim_vo, k_global_scale, v_global_scale, layout.page_size)

    def struct(self) -> PagedCacheStruct:
        s = PagedCacheStruct()
        s.k_data, s.v_data = self.k_data.data_ptr(), self.v_data.data_ptr()
        s.k_sf, s.v_sf = self.k_sf.data_ptr(), self.v_sf.data_ptr()
        for w, pre in (("k_data", "k"), ("v_data", "v"), ("k_sf", "k_sf"),
                       ("v_sf", "v_sf")):
            sp, ss, sh = self.strides[w]
            setattr(s, pre + "_stride_page", sp)
            setattr(s, pre + "_stride_slot", ss)
            setattr(s, pre + "_stride_head", sh)
        s.num_pages, s.page_size = self.num_pages, self.page_size
        s.num_kv_heads = self.num_kv_heads
        s.head_dim_qk, s.head_dim_vo = self.head_dim_qk, self.head_dim_vo
        s.k_global_scale, s.v_global_scale = self.k_global_scale, self.v_global_scale
        return s

    def host_copy(self):
        return {w: getattr(self, w).cpu() for w in ("k_data", "v_data", "k_sf", "v_sf")}


def nvfp4kv_quantize_append(cache: PagedCache, k: torch.Tensor, v: torch.Tensor,
                            batch_idx, positions, kv_indices, kv_indptr,
                            last_page_len, device_flags=None, stream=None):
    """Quantise bf16 K [nnz, Hkv, Dk] / V [nnz, Hkv, Dv] into their pages."""
    L = _lib.load()
    s = cache.struct()
    nnz = int(k.shape[0]) if k.numel() else 0
    st = L.nvfp4kv_quantize_append(
        C.byref(s), _ptr(k), k.stride(0) if k.dim() == 3 else 0,
        k.stride(1) if k.dim() == 3 else 0, _ptr(v), v.stride(0) if v.dim() == 3 else 0,
        v.stride(1) if v.dim() == 3 else 0, nnz, _ptr(batch_idx), _ptr(positions),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(last_page_len),
        int(kv_indptr.numel()) - 1, _ptr(device_flags), _stream(stream))
    check(st, "nvfp4kv_quantize_append")


def nvfp4kv_dequantize_paged(cache: PagedCache, page_ids, k_out=None, v_out=None,
                             want_k=True, want_v=True, device_flags=None, stream=None):
    """Dequantise the listed pages to float32: returns (k, v), each
    [len(page_ids), page_size, Hkv, D] (or None when not wanted)."""
    L = _lib.load()
    n = int(page_ids.numel())
    dev = cache.k_data.device
    if want_k and k_out is None:
        k_out = torch.empty((n, cache.page_size, cache.num_kv_heads, cache.head_dim_qk),
                            dtype=torch.float32, device=dev)
    if want_v and v_out is None:
        v_out = torch.empty((n, cache.page_size, cache.num_kv_heads, cache.head_dim_vo),
                            dtype=torch.float32, device=dev)
    s = cache.struct()
    st = L.nvfp4kv_dequantize_paged(C.byref(s), _ptr(page_ids), n,
                                    _ptr(k_out if want_k else None),
                                    _ptr(v_out if want_v else None), _ptr(device_flags),
                                    _stream(stream))
    check(st, "nvfp4kv_dequantize_paged")
    return (k_out if want_k else None), (v_out if want_v else None)


class Plan:
    """A decode plan: the C plan_info, its pinned host work list and the
    device workspace it was uploaded into (and the live length array it
    reads, kept alive with it)."""

    def __init__(self, info: PlanInfo, host: torch.Tensor, workspace: torch.Tensor,
                 live=None):
        self.info, self.host, self.workspace, self.live = info, host, workspace, live

    def __getattr__(self, name):
        return getattr(self.info, name)

    def partial_views(self):
        ws, i = self.workspace, self.info
        n, dv = i.num_partials, i.head_dim_vo
        lse = ws[i.off_partial_lse: i.off_partial_lse + 4 * n].view(torch.float32)
        o = ws[i.off_partial_o: i.off_partial_o + 4 * n * dv].view(torch.float32).view(n, dv)
        e = i.total_qo_rows * i.num_qo_heads
        mi = ws[i.off_merge_indptr: i.off_merge_indptr + 4 * (e + 1)].view(torch.int32)
        return o, lse, mi


def _host_i32(t) -> torch.Tensor:
    return torch.as_tensor(t, dtype=torch.int32).cpu().contiguous()


def nvfp4kv_decode_plan(qo_indptr, kv_indptr, last_page_len, num_qo_heads: int,
                        num_kv_heads: int, head_dim_qk: int, head_dim_vo: int,
                        page_size: int = 16, causal: bool = False,
                        disable_split: bool = False, max_splits: int = 0,
                        force_chunk_tokens: int = 0, kernel: int = 0, num_sms: int = 0,
                        ctas_per_sm: int = 0, device: Optional[int] = None,
                        allocate: bool = True, reuse: Optional[Plan] = None,
                        device_last_page_len: Optional[torch.Tensor] = None,
                        out_dtype: torch.dtype = torch.bfloat16, stream=None) -> Plan:
    """Plan from host copies of the indptrs; allocates the pinned host buffer
    and the device workspace (torch) and uploads the work list.  With
    ``reuse`` the plan is written into that plan's buffers when they are big
    enough (one library call, no allocation).  ``device_last_page_len`` (an
    int32 device tensor [batch]) makes every run read the current last page
    lengths from it (the plan stays valid while page and query counts do).
    ``out_dtype`` is torch.bfloat16 (default) or torch.float16.  ``kernel``:
    0 auto, 1 tensor-core mma.sync, 2 CUDA-core, 3 tcgen05 (head dims 128),
    4 FP4 query and probabilities (at most 8 query rows per kv head, head
    dims 64 or 128; two launches per run), as in nvfp4kv.h."""
    if out_dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float16")
    L = _lib.load()
    qo, kv, lp = _host_i32(qo_indptr), _host_i32(kv_indptr), _host_i32(last_page_len)
    batch = int(kv.numel()) - 1
    opts = PlanOptions(int(causal), int(disable_split), int(max_splits),
                       int(force_chunk_tokens), int(kernel), int(num_sms), int(ctas_per_sm),
                       1 if out_dtype == torch.float16 else 0,
                       None if device_last_page_len is None
                       else device_last_page_len.data_ptr())
    info = PlanInfo()
    dev = -1 if device is None else int(device)
    args = (qo.data_ptr(), kv.data_ptr(), lp.data_ptr(), batch, num_qo_heads, num_kv_heads,
            head_dim_qk, head_dim_vo, page_size, C.byref(opts), dev)
    if reuse is not None and reuse.workspace is not None:
        st = L.nvfp4kv_decode_plan(*args, _ptr(reuse.host), reuse.host.numel(),
                                   _ptr(reuse.workspace), reuse.workspace.numel(),
                                   _stream(stream), C.byref(info))
        if st == _lib.OK:
            return Plan(info, reuse.host, reuse.workspace, device_last_page_len)
        if st != _lib.ERR_WORKSPACE_TOO_SMALL:
            check(st, "nvfp4kv_decode_plan")
    st = L.nvfp4kv_decode_plan(*args, None, 0, None, 0, None, C.byref(info))
    if st not in (_lib.OK, _lib.ERR_WORKSPACE_TOO_SMALL):
        check(st, "nvfp4kv_decode_plan")
    nhost = max(int(info.plan_host_bytes), 16)
    pin = allocate and torch.cuda.is_available()
    host = torch.empty(nhost, dtype=torch.uint8, pin_memory=pin)
    if not allocate:
        st = L.nvfp4kv_decode_plan(*args, _ptr(host), nhost, None, 0, None, C.byref(info))
        check(st, "nvfp4kv_decode_plan")
        return Plan(info, host, None, device_last_page_len)
    ws = torch.empty(max(int(info.workspace_bytes), 256), dtype=torch.uint8,
                     device="cuda" if device is None else "cuda:%d" % device)
    st = L.nvfp4kv_decode_plan(*args, _ptr(host), nhost, _ptr(ws), ws.numel(),
                               _stream(stream), C.byref(info))
    check(st, "nvfp4kv_decode_plan")
    return Plan(info, host, ws, device_last_page_len)


def _outputs(plan: Plan, out, lse, device):
    rows, hq, dv = plan.info.total_qo_rows, plan.info.num_qo_heads, plan.info.head_dim_vo
    if out is None:
        dt = torch.float16 if plan.info.out_dtype == 1 else torch.bfloat16
        out = torch.empty((rows, hq, dv), dtype=dt, device=device)
    if lse is None:
        lse = torch.empty((rows, hq), dtype=torch.float32, device=device)
    return out, lse


def _run(fn, name, plan, q, cache, kv_indices, sm_scale, out, lse, stream):
    out, lse = _outputs(plan, out, lse, q.device)
    s = cache.struct()
    st = fn(C.byref(plan.info), _ptr(q), q.stride(0), q.stride(1), C.byref(s),
            _ptr(kv_indices), float(sm_scale or 0.0), _ptr(plan.workspace),
            plan.workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    check(st, name)
    return out, lse


def nvfp4kv_decode_run(plan: Plan, q: torch.Tensor, cache: PagedCache, kv_indices,
                       sm_scale: float = 0.0, out=None, lse=None, stream=None):
    """Attention (+ merge when split).  Returns (out bf16 [rows,Hq,Dv], lse)."""
    return _run(_lib.load().nvfp4kv_decode_run, "nvfp4kv_decode_run", plan, q, cache,
                kv_indices, sm_scale, out, lse, stream)


def nvfp4kv_decode_attend(plan: Plan, q: torch.Tensor, cache: PagedCache, kv_indices,
                          sm_scale: float = 0.0, out=None, lse=None, stream=None):
    return _run(_lib.load().nvfp4kv_decode_attend, "nvfp4kv_decode_attend", plan, q,
                cache, kv_indices, sm_scale, out, lse, stream)


def nvfp4kv_decode_append_run(plan: Plan, new_k: torch.Tensor, new_v: torch.Tensor,
                              q: torch.Tensor, cache: PagedCache, kv_indices,
                              sm_scale: float = 0.0, out=None, lse=None, stream=None):
    """Quantise the step's new tokens (bf16 [rows, Hkv, D], row-aligned with
    q) into the cache and run the attention, in one launch."""
    out, lse = _outputs(plan, out, lse, q.device)
    s = cache.struct()
    st = _lib.load().nvfp4kv_decode_append_run(
        C.byref(plan.info), _ptr(new_k), new_k.stride(0), new_k.stride(1), _ptr(new_v),
        new_v.stride(0), new_v.stride(1), _ptr(q), q.stride(0), q.stride(1), C.byref(s),
        _ptr(kv_indices), float(sm_scale or 0.0), _ptr(plan.workspace),
        plan.workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    check(st, "nvfp4kv_decode_append_run")
    return out, lse


def nvfp4kv_decode_merge(plan: Plan, out, lse, stream=None):
    st = _lib.load().nvfp4kv_decode_merge(C.byref(plan.info), _ptr(plan.workspace),
                                          plan.workspace.numel(), _ptr(out), _ptr(lse),
                                          _stream(stream))
    check(st, "nvfp4kv_decode_merge")
    return out, lse


def nvfp4kv_merge_states(o_partial: torch.Tensor, lse_partial: torch.Tensor,
                         merge_indptr: torch.Tensor, out=None, lse=None, stream=None):
    """Merge float32 partial states o_partial [P, Dv], lse_partial [P] over
    the ranges of merge_indptr [E+1]; returns (out bf16 [E, Dv], lse [E])."""
    E = int(merge_indptr.numel()) - 1
    dv = int(o_partial.shape[-1])
    if out is None:
        out = torch.empty((E, dv), dtype=torch.bfloat16, device=o_partial.device)
    if lse is None:
        lse = torch.empty((E,), dtype=torch.float32, device=o_partial.device)
    st = _lib.load().nvfp4kv_merge_states(_ptr(o_partial), _ptr(lse_partial),
                                          _ptr(merge_indptr), E, dv, _ptr(out), _ptr(lse),
                                          _stream(stream))
    check(st, "nvfp4kv_merge_states")
    return out, lse


def nvfp4kv_workspace_flags(plan: Plan, clear: bool = False, stream=None) -> int:
    flags = C.c_uint32(0)
    st = _lib.load().nvfp4kv_workspace_flags(C.byref(plan.info), _ptr(plan.workspace),
                                             C.byref(flags), int(clear), _stream(stream))
    if st not in (_lib.OK, _lib.ERR_DEVICE_CHECK):
        check(st, "nvfp4kv_workspace_flags")
    return int(flags.value)


def nvfp4kv_decode_run_static(plan: Plan, q: torch.Tensor, cache: PagedCache, kv_indices,
                              sm_scale: float = 0.0, out=None, lse=None, stream=None):
    """nvfp4kv_decode_run without a caller workspace: the library's fixed
    16 MiB array serves as the workspace (for callers that cannot allocate
    device memory).  ``plan`` is a host-only plan
    (``nvfp4kv_decode_plan(..., allocate=False)``); ``out``/``lse`` should be
    passed by such callers (allocated here only when omitted)."""
    out, lse = _outputs(plan, out, lse, q.device)
    s = cache.struct()
    st = _lib.load().nvfp4kv_decode_run_static(
        C.byref(plan.info), _ptr(plan.host), _ptr(q), q.stride(0), q.stride(1), C.byref(s),
        _ptr(kv_indices), float(sm_scale or 0.0), _ptr(out), _ptr(lse), _stream(stream))
    check(st, "nvfp4kv_decode_run_static")
    return out, lse


def default_sm_scale(head_dim_qk: int) -> float:
    return 1.0 / math.sqrt(head_dim_qk)


def nvfp4kv_static_workspace_flags(plan: Plan, clear: bool = False, stream=None) -> int:
    """The flag word of the static workspace after nvfp4kv_decode_run_static."""
    flags = C.c_uint32(0)
    st = _lib.load().nvfp4kv_static_workspace_flags(C.byref(plan.info), C.byref(flags),
                                                    int(clear), _stream(stream))
    if st not in (_lib.OK, _lib.ERR_DEVICE_CHECK):
        check(st, "nvfp4kv_static_workspace_flags")
    return int(flags.value)
