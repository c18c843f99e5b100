"""Host-only checks of the C-ABI library: it builds and loads, exports every
function the header declares, validates arguments before touching CUDA, and
plans split-KV work with the stated invariants (device queries replaced by
the num_sms / ctas_per_sm overrides, so no GPU is needed)."""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import _lib
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

UNIT_DTYPE = np.dtype([(n, "<i4") for n in (
    "b", "h_kv", "page_begin", "num_pages", "tok_begin", "kv_len", "qo_begin", "qo_len",
    "split", "num_splits", "partial_base", "pair")])


def test_library_exports_header_symbols():
    L = _lib.load()
    names = _lib.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    for n in ("nvfp4kv_quantize_append", "nvfp4kv_decode_plan", "nvfp4kv_decode_run",
              "nvfp4kv_merge_states"):
        assert n in names


def test_status_strings():
    L = _lib.load()
    assert L.nvfp4kv_status_string(0) == b"ok"
    assert L.nvfp4kv_status_string(3) == b"workspace too small"
    assert L.nvfp4kv_status_string(99) == b"unknown status"


def plan(batch, **kw):
    c = batch.cfg
    args = dict(num_sms=152, ctas_per_sm=3, allocate=False, causal=c.causal)
    args.update(kw)
    return N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk,
                                 c.head_dim_vo, **args)


def units_of(p):
    raw = p.host.numpy()[: p.info.num_units * UNIT_DTYPE.itemsize]
    return np.frombuffer(raw.tobytes(), dtype=UNIT_DTYPE)


def merge_indptr_of(p):
    i = p.info
    off = i.off_merge_indptr - i.off_units
    e = i.total_qo_rows * i.num_qo_heads
    return np.frombuffer(p.host.numpy()[off: off + 4 * (e + 1)].tobytes(), "<i4")


def check_cover(batch, p):
    """Every (request, kv head) page range is covered once, in 16-token chunks."""
    u = units_of(p)
    c = batch.cfg
    kvp = batch.kv_indptr.tolist()
    P = batch.page_size
    for b in range(c.batch):
        for h in range(c.num_kv_heads):
            sel = u[(u["b"] == b) & (u["h_kv"] == h)]
            sel = sel[np.argsort(sel["split"])]
            assert len(sel) == sel["num_splits"][0]
            pos = kvp[b]
            for k, x in enumerate(sel):
                assert x["split"] == k and x["page_begin"] == pos
                assert x["tok_begin"] == (pos - kvp[b]) * P and x["tok_begin"] % 16 == 0
                assert x["kv_len"] == batch.kv_lens[b]
                pos += x["num_pages"]
            assert pos == kvp[b + 1]
    return u


@pytest.mark.parametrize("page_size", [16, 1])
@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_plan_covers_all_pages(name, page_size):
    batch = W.make_batch(W.WORKLOADS[name]) if name != "prefix_cache_extend" else None
    if batch is None:  # the big extend batch: same page table, cheaper draw
        cfg = W.WORKLOADS[name]
        batch = W.make_batch(W.custom_workload(
            kv_lens=[2000 + 997 * i for i in range(32)], qo_len=16, num_qo_heads=32,
            num_kv_heads=8, causal=True, shared_prefix_tokens=1024, seed=cfg.seed,
            batch=32))
    if page_size == 1:
        batch = W.with_page_size_one(batch)
    p = plan(batch, page_size=batch.page_size)
    u = check_cover(batch, p)
    i = p.info
    ctas = i.num_units * i.row_blocks
    pairs = batch.cfg.batch * batch.cfg.num_kv_heads
    if i.split:
        # one wave: the grid fits the resident CTA slots
        assert ctas <= 152 * 3
        assert i.num_partials == sum(
            n * batch.cfg.num_qo_heads * s for n, s in zip(
                [batch.cfg.qo_len] * batch.cfg.batch,
                [u[(u["b"] == b) & (u["h_kv"] == 0)]["num_splits"][0]
                 for b in range(batch.cfg.batch)]))
        mi = merge_indptr_of(p)
        assert mi[0] == 0 and mi[-1] == i.num_partials and np.all(np.diff(mi) >= 1)
    else:
        assert i.num_units == pairs
    if ctas > i.num_sms * i.ctas_per_sm:  # more than one wave: longest units first
        assert list(u["num_pages"]) == sorted(u["num_pages"], reverse=True)


def test_plan_orders_multi_wave_grids_longest_first():
    # 16-token chunks of requests of different lengths: many waves, and the
    # last unit of each request is shorter than the rest
    batch = W.make_batch(W.WORKLOADS["batched_decode"])
    p = plan(batch, force_chunk_tokens=64)
    u = check_cover(batch, p)
    assert p.info.num_units * p.info.row_blocks > 152 * 3
    assert len(set(u["num_pages"])) > 1
    assert list(u["num_pages"]) == sorted(u["num_pages"], reverse=True)
    # one-wave grids keep the order they are built in: request, kv head, split
    q = plan(batch)
    v = units_of(q)
    assert q.info.num_units * q.info.row_blocks <= 152 * 3
    key = [(int(b), int(h), int(s)) for b, h, s in zip(v["b"], v["h_kv"], v["split"])]
    assert key == sorted(key)


def test_plan_long_context_splits_in_one_wave():
    batch = W.make_batch(W.WORKLOADS["long_context_decode"])
    p = plan(batch)
    assert p.info.split == 1 and p.info.chunk_pages * 16 % 16 == 0
    assert p.info.num_units <= 152 * 3 and p.info.num_units >= 152 * 3 * 0.8
    p2 = plan(batch, disable_split=True)
    assert p2.info.split == 0 and p2.info.num_units == 32
    p3 = plan(batch, force_chunk_tokens=2048)
    assert p3.info.chunk_pages == 128 and p3.info.max_units_per_request == 17
    p4 = plan(batch, max_splits=4)
    assert p4.info.max_units_per_request <= 4
    p5 = plan(batch, force_chunk_tokens=16)
    check_cover(batch, p5)
    assert p5.info.max_units_per_request == 2049


def test_plan_small_batch_does_not_split():
    batch = W.make_batch(W.WORKLOADS["tiny_decode"])
    p = plan(batch)
    assert p.info.split == 0 and p.info.num_units == 2 and p.info.rows_per_block == 8


def test_plan_rows_per_block():
    batch = W.make_batch(W.custom_workload(kv_lens=(40, 70), qo_len=3, num_qo_heads=8,
                                           num_kv_heads=2, causal=True))
    p = plan(batch)  # 3 positions x 4 heads = 12 rows -> one 16-row block
    assert p.info.rows_per_block == 16 and p.info.row_blocks == 1


def plan_status(qo, kv, last, hq=4, hkv=1, dk=128, dv=128, ps=16, **opts):
    L = _lib.load()
    o = _lib.PlanOptions(0, 0, 0, opts.get("force", 0), 0, 152, 3)
    info = _lib.PlanInfo()
    qo, kv, last = (torch.tensor(x, dtype=torch.int32) for x in (qo, kv, last))
    return L.nvfp4kv_decode_plan(qo.data_ptr(), kv.data_ptr(), last.data_ptr(),
                                 len(kv) - 1, hq, hkv, dk, dv, ps, C.byref(o), -1, None, 0,
                                 None, 0, None, C.byref(info))


@pytest.mark.parametrize("case,status", [
    (dict(hq=6, hkv=4), _lib.ERR_INVALID_ARGUMENT),
    (dict(ps=8), _lib.ERR_UNSUPPORTED),
    (dict(dk=96, dv=96), _lib.ERR_UNSUPPORTED),
    (dict(dk=128, dv=256), _lib.ERR_UNSUPPORTED),
    (dict(last=[0, 5]), _lib.ERR_INVALID_ARGUMENT),
    (dict(last=[17, 5]), _lib.ERR_INVALID_ARGUMENT),
    (dict(qo=[0, 2, 3], kv=[0, 1, 10], last=[1, 5]), _lib.ERR_INVALID_ARGUMENT),  # L < n
    (dict(qo=[1, 2, 3]), _lib.ERR_INVALID_ARGUMENT),
    (dict(kv=[0, 3, 2]), _lib.ERR_INVALID_ARGUMENT),
    (dict(force=24), _lib.ERR_INVALID_ARGUMENT),
])
def test_plan_rejects(case, status):
    args = dict(qo=[0, 1, 2], kv=[0, 3, 10], last=[5, 4])
    args.update(case)
    qo, kv, last = args.pop("qo"), args.pop("kv"), args.pop("last")
    assert plan_status(qo, kv, last, **args) == status
    assert _lib.load().nvfp4kv_last_error_detail()


def test_plan_size_query_reports_sizes():
    assert plan_status([0, 1, 2], [0, 3, 10], [5, 4]) == _lib.ERR_WORKSPACE_TOO_SMALL


def fake_cache(dk=128, dv=128, **over):
    s = _lib.PagedCacheStruct()
    s.k_data, s.v_data, s.k_sf, s.v_sf = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    H = 2
    for pre, row in (("k", dk // 2), ("v", dv // 2), ("k_sf", dk // 16), ("v_sf", dv // 16)):
        setattr(s, pre + "_stride_page", 16 * H * row)
        setattr(s, pre + "_stride_slot", row)
        setattr(s, pre + "_stride_head", 16 * row)
    s.num_pages, s.page_size, s.num_kv_heads = 10, 16, H
    s.head_dim_qk, s.head_dim_vo = dk, dv
    s.k_global_scale = s.v_global_scale = 1.0
    for k, v in over.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("over,status", [
    (dict(k_data=None), _lib.ERR_INVALID_ARGUMENT),
    (dict(page_size=8), _lib.ERR_UNSUPPORTED),
    (dict(k_stride_slot=40), _lib.ERR_INVALID_ARGUMENT),        # not a multiple of 16
    (dict(v_stride_head=32), _lib.ERR_INVALID_ARGUMENT),        # overlaps a 64-byte row
    (dict(k_sf_stride_slot=4), _lib.ERR_INVALID_ARGUMENT),      # overlaps / misaligned
    (dict(v_data=(2 << 20) + 8), _lib.ERR_INVALID_ARGUMENT),    # misaligned base
    (dict(head_dim_qk=100), _lib.ERR_UNSUPPORTED),
    (dict(k_global_scale=0.0), _lib.ERR_INVALID_ARGUMENT),
    (dict(v_global_scale=float("inf")), _lib.ERR_INVALID_ARGUMENT),
])
def test_append_rejects_bad_cache(over, status):
    L = _lib.load()
    s = fake_cache(**over)
    buf = 1 << 24
    st = L.nvfp4kv_quantize_append(C.byref(s), buf, 256, 128, buf, 256, 128, 1, buf, buf,
                                   buf, buf, buf, 1, None, None)
    assert st == status


def test_append_rejects_bad_inputs_and_accepts_empty():
    L = _lib.load()
    s = fake_cache()
    buf = 1 << 24
    assert L.nvfp4kv_quantize_append(C.byref(s), buf, 256, 128, buf, 256, 128, 0, None, None,
                                     None, None, None, 1, None, None) == 0
    assert L.nvfp4kv_quantize_append(C.byref(s), buf + 2, 256, 128, buf, 256, 128, 1, buf,
                                     buf, buf, buf, buf, 1, None, None) == 1
    assert L.nvfp4kv_quantize_append(C.byref(s), buf, 250, 128, buf, 256, 128, 1, buf, buf,
                                     buf, buf, buf, 1, None, None) == 1
    assert L.nvfp4kv_quantize_append(C.byref(s), None, 256, 128, buf, 256, 128, 1, buf, buf,
                                     buf, buf, buf, 1, None, None) == 1


def test_run_rejects_mismatched_cache_and_bad_plan():
    L = _lib.load()
    batch = W.make_batch(W.WORKLOADS["tiny_decode"])
    p = plan(batch)
    s = fake_cache(num_kv_heads=1)
    buf = 1 << 24
    ws = 1 << 26
    args = lambda info, cache: (C.byref(info), buf, 512, 128, C.byref(cache), buf, 0.0, ws,
                                p.info.workspace_bytes, buf, buf, None)
    s2 = fake_cache()  # 2 kv heads, plan has 1
    assert L.nvfp4kv_decode_run(*args(p.info, s2)) == _lib.ERR_PLAN_MISMATCH
    bad = _lib.PlanInfo()
    assert L.nvfp4kv_decode_run(*args(bad, s)) == _lib.ERR_INVALID_ARGUMENT
    s3 = fake_cache(num_kv_heads=1, head_dim_qk=256, head_dim_vo=64)
    assert L.nvfp4kv_decode_run(*args(p.info, s3)) == _lib.ERR_UNSUPPORTED
    st = L.nvfp4kv_decode_run(C.byref(p.info), buf, 512, 128, C.byref(s), buf, 0.0, ws,
                              16, buf, buf, None)
    assert st == _lib.ERR_WORKSPACE_TOO_SMALL
    st = L.nvfp4kv_decode_run(C.byref(p.info), buf + 4, 512, 128, C.byref(s), buf, 0.0, ws,
                              p.info.workspace_bytes, buf, buf, None)
    assert st == _lib.ERR_INVALID_ARGUMENT


def test_merge_states_rejects():
    L = _lib.load()
    buf = 1 << 24
    assert L.nvfp4kv_merge_states(buf, buf, buf, 4, 100, buf, buf, None) == _lib.ERR_UNSUPPORTED
    assert L.nvfp4kv_merge_states(buf, buf, buf, -1, 128, buf, buf, None) == 1
    assert L.nvfp4kv_merge_states(None, buf, buf, 4, 128, buf, buf, None) == 1
    assert L.nvfp4kv_merge_states(None, None, None, 0, 128, None, None, None) == 0


@pytest.mark.parametrize("qo_len,rows", [(1, 16), (4, 16), (7, 32), (16, 64), (20, 64)])
def test_plan_tcgen05_rows_and_tiles(qo_len, rows):
    """kernel=3 plans N = 16 / 32 / 64 query rows per CTA (G * n rounded up,
    64 at most) and, when it splits on its own, whole 8-page tiles per unit."""
    batch = W.make_batch(W.custom_workload(batch=3, qo_len=qo_len, num_qo_heads=8,
                                           num_kv_heads=2, kv_lens=(40, 3000, 9000),
                                           causal=qo_len > 1))
    p = plan(batch, kernel=3, ctas_per_sm=1)
    assert p.info.kernel == 3 and p.info.rows_per_block == rows
    assert p.info.row_blocks == -(-4 * qo_len // rows)
    check_cover(batch, p)
    if p.info.split:
        max_np = int(np.diff(batch.kv_indptr.numpy()).max())
        assert p.info.chunk_pages % 8 == 0 or p.info.chunk_pages == max_np


def test_plan_tcgen05_rejects_other_dims():
    batch = W.make_batch(W.custom_workload(batch=1, head_dim_qk=256, head_dim_vo=128,
                                           kv_lens=(100,)))
    with pytest.raises(N.NvFp4KvError):
        plan(batch, kernel=3)


def test_plan_auto_kernel_choice():
    """Auto picks tcgen05 for many query rows per kv head at head dims 128
    (extend) and the mma.sync kernel for decode or other head dims."""
    ext = W.make_batch(W.custom_workload(batch=2, qo_len=16, num_qo_heads=8, num_kv_heads=2,
                                         kv_lens=(100, 900), causal=True))
    assert plan(ext, ctas_per_sm=1).info.kernel == 3
    dec = W.make_batch(W.custom_workload(batch=2, qo_len=1, num_qo_heads=8, num_kv_heads=2,
                                         kv_lens=(100, 900)))
    assert plan(dec).info.kernel == 1
    wide = W.make_batch(W.custom_workload(batch=2, qo_len=16, num_qo_heads=8, num_kv_heads=2,
                                          head_dim_qk=256, head_dim_vo=256,
                                          kv_lens=(100, 900), causal=True))
    assert plan(wide).info.kernel == 1


def test_dequantize_rejects_bad_arguments_and_accepts_empty():
    """nvfp4kv_dequantize_paged validates on the host before any launch."""
    L = _lib.load()
    s = fake_cache()
    buf = 1 << 24
    # nothing to do: no ids, or no output wanted
    assert L.nvfp4kv_dequantize_paged(C.byref(s), None, 0, buf, buf, None, None) == 0
    assert L.nvfp4kv_dequantize_paged(C.byref(s), buf, 4, None, None, None, None) == 0
    assert L.nvfp4kv_dequantize_paged(C.byref(s), buf, -1, buf, buf, None, None) == \
        _lib.ERR_INVALID_ARGUMENT
    assert L.nvfp4kv_dequantize_paged(C.byref(s), None, 4, buf, buf, None, None) == \
        _lib.ERR_INVALID_ARGUMENT
    assert L.nvfp4kv_dequantize_paged(C.byref(s), buf, 4, buf + 4, None, None, None) == \
        _lib.ERR_INVALID_ARGUMENT  # output not 16-byte aligned
    bad = fake_cache(page_size=8)
    assert L.nvfp4kv_dequantize_paged(C.byref(bad), buf, 4, buf, buf, None, None) == \
        _lib.ERR_UNSUPPORTED


def test_plan_page_size_one_matches_sixteen():
    """The same batch over 1-token pages plans the same units in tokens: the
    unit token ranges, splits and kv lengths agree with the 16-token plan and
    each unit holds 16 times the pages."""
    batch = W.make_batch(W.WORKLOADS["batched_decode"])
    b1 = W.with_page_size_one(batch)
    p16, p1 = plan(batch), plan(b1, page_size=1)
    u16, u1 = units_of(p16), units_of(p1)
    assert p1.info.num_units == p16.info.num_units
    for f in ("b", "h_kv", "tok_begin", "kv_len", "split", "num_splits", "partial_base"):
        assert np.array_equal(u16[f], u1[f]), f
    tok16 = np.minimum(u16["num_pages"] * 16, u16["kv_len"] - u16["tok_begin"])
    assert np.array_equal(tok16, u1["num_pages"])
    check_cover(b1, p1)


def test_plan_rejects_other_page_sizes_and_dtypes():
    batch = W.make_batch(W.WORKLOADS["tiny_decode"])
    for ps in (8, 32, 0):
        with pytest.raises(N.NvFp4KvError) as e:
            plan(batch, page_size=ps)
        assert e.value.status == _lib.ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        plan(batch, out_dtype=torch.float32)
    p = plan(batch, out_dtype=torch.float16)
    assert p.info.out_dtype == 1


def test_plan_fp4qp_row_max_region():
    """kernel=4 (FP4 query and probabilities) plans the mma.sync work list and
    a row-maximum region of rows x Hq x units-per-request floats after the
    partial states; it takes one block of at most 8 query rows and head dims
    64 or 128."""
    batch = W.make_batch(W.custom_workload(batch=3, qo_len=1, num_qo_heads=8, num_kv_heads=2,
                                           kv_lens=(40, 3000, 9000)))
    p = plan(batch, kernel=4)
    i = p.info
    assert i.kernel == 4 and i.rows_per_block == 8
    check_cover(batch, p)
    assert i.off_row_max >= i.off_partial_o and i.off_row_max % 256 == 0
    need = i.total_qo_rows * i.num_qo_heads * max(i.max_units_per_request, 1) * 4
    assert i.workspace_bytes >= i.off_row_max + need
    assert plan(batch, kernel=1).info.off_row_max == 0
    ext = W.make_batch(W.custom_workload(batch=2, qo_len=4, num_qo_heads=8, num_kv_heads=2,
                                         kv_lens=(100, 900), causal=True))
    with pytest.raises(N.NvFp4KvError):      # 16 rows per kv head
        plan(ext, kernel=4)
    wide = W.make_batch(W.custom_workload(batch=1, head_dim_qk=256, head_dim_vo=256,
                                          kv_lens=(100,)))
    with pytest.raises(N.NvFp4KvError):
        plan(wide, kernel=4)
