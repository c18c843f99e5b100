"""The allocation-free attention entry point (nvfp4kv_decode_run_static).

It is for callers that cannot allocate device memory where they run attention
(device memory fully reserved up front, a host framework without scratch
buffers, or a path that must not call cudaMalloc): the library's fixed 16 MiB
array is the workspace.  Its output must match the allocating entry point's,
on two calls in a row (the array keeps the previous call's contents), and a
plan that needs more than the array holds must be rejected before anything
runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import gpu_harness as H
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import _lib
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def host_plan(batch, **kw):
    c = batch.cfg
    return N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 causal=c.causal, allocate=False, **kw)


@pytest.mark.parametrize("qo_len,causal", [(1, False), (5, True)])
def test_static_workspace_matches_allocating_entry_point(qo_len, causal):
    batch = W.make_batch(W.custom_workload(
        seed=31, batch=4, kv_lens=(37, 300, 1000, 2500), qo_len=qo_len, num_qo_heads=16,
        num_kv_heads=4, causal=causal))
    # the allocating entry point (caller workspace), split into 64-token chunks
    g = H.GpuCase(batch, force_chunk_tokens=64)
    assert g.plan.info.split == 1
    ref_out, ref_lse = g.run()
    plan = host_plan(batch, force_chunk_tokens=64)
    assert plan.workspace is None and plan.info.split == 1
    rows, c = int(batch.qo_indptr[-1]), batch.cfg
    for call in range(2):
        out = torch.full((rows, c.num_qo_heads, c.head_dim_vo), float("nan"),
                         dtype=torch.bfloat16, device="cuda")
        lse = torch.full((rows, c.num_qo_heads), float("nan"), device="cuda")
        N.nvfp4kv_decode_run_static(plan, g.q, g.cache, g.kv_indices, batch.sm_scale,
                                    out=out, lse=lse)
        torch.cuda.synchronize()
        # same tolerance as the parity tests: 5e-3 beyond the bf16 rounding
        H.compare(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy())


def test_static_workspace_rejects_plans_beyond_its_size():
    batch = W.make_batch(W.WORKLOADS["long_context_decode"])
    plan = host_plan(batch, force_chunk_tokens=16)      # 2049 splits per request
    assert plan.info.workspace_bytes > (16 << 20)
    g_cache = N.PagedCache.allocate(batch.cache_layout(), 1.0, 1.0)
    q = batch.q.cuda()
    kvi = torch.as_tensor(batch.kv_indices).to(torch.int32).cuda()
    out = torch.full((4, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(N.NvFp4KvError) as err:
        N.nvfp4kv_decode_run_static(plan, q, g_cache, kvi, batch.sm_scale, out=out,
                                    lse=torch.zeros((4, 32), device="cuda"))
    assert err.value.status == _lib.ERR_WORKSPACE_TOO_SMALL
    assert "16 MiB" in err.value.detail
    torch.cuda.synchronize()
    assert torch.all(out.float() == 7.0)   # nothing ran


def test_static_workspace_reports_a_bad_page_id():
    """A page id outside the pool sets the bad-page flag in the static
    array's flag word; nvfp4kv_static_workspace_flags reads it (and clears
    it), and the next good call reports a clean word."""
    batch = W.make_batch(W.custom_workload(seed=33, batch=2, kv_lens=(37, 300),
                                           num_qo_heads=8, num_kv_heads=2))
    g = H.GpuCase(batch)
    plan = host_plan(batch)
    rows, c = int(batch.qo_indptr[-1]), batch.cfg
    out = torch.empty((rows, c.num_qo_heads, c.head_dim_vo), dtype=torch.bfloat16,
                      device="cuda")
    bad = g.kv_indices.clone()
    bad[2] = batch.num_pages + 11
    N.nvfp4kv_decode_run_static(plan, g.q, g.cache, bad, batch.sm_scale, out=out)
    assert N.nvfp4kv_static_workspace_flags(plan, clear=True) & _lib.FLAG_BAD_PAGE_INDEX
    assert N.nvfp4kv_static_workspace_flags(plan) == 0
    N.nvfp4kv_decode_run_static(plan, g.q, g.cache, g.kv_indices, batch.sm_scale, out=out)
    assert N.nvfp4kv_static_workspace_flags(plan) == 0
    assert bool(torch.isfinite(out.float()).all())


def test_static_workspace_rejected_call_leaves_the_array_alone():
    """A call that fails argument checks enqueues nothing: the flag word the
    previous call left is still there."""
    batch = W.make_batch(W.custom_workload(seed=34, batch=2, kv_lens=(40, 90),
                                           num_qo_heads=4, num_kv_heads=1))
    g = H.GpuCase(batch)
    plan = host_plan(batch)
    bad = g.kv_indices.clone()
    bad[0] = -3
    out = torch.empty((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    N.nvfp4kv_decode_run_static(plan, g.q, g.cache, bad, batch.sm_scale, out=out)
    torch.cuda.synchronize()
    n = g.q.numel()
    q_off = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")[1:1 + n].view(g.q.shape)
    q_off.copy_(g.q)
    with pytest.raises(N.NvFp4KvError) as err:   # q misaligned: rejected on the host
        N.nvfp4kv_decode_run_static(plan, q_off, g.cache, g.kv_indices, batch.sm_scale,
                                    out=out)
    assert err.value.status == _lib.ERR_INVALID_ARGUMENT
    assert N.nvfp4kv_static_workspace_flags(plan, clear=True) & _lib.FLAG_BAD_PAGE_INDEX


def test_fp4qp_static_entry_point():
    """The allocation-free entry point runs both launches of a kernel-4 plan
    (the row maxima in its fixed array) and gives the allocating entry
    point's outputs bit for bit."""
    batch = W.make_batch(W.custom_workload(seed=31, batch=4, kv_lens=(37, 300, 1000, 2500),
                                           qo_len=1, num_qo_heads=16, num_kv_heads=4))
    g = H.GpuCase(batch, kernel=4, force_chunk_tokens=64)
    ref_out, ref_lse = g.run()
    plan = host_plan(batch, kernel=4, force_chunk_tokens=64)
    assert plan.info.kernel == 4 and plan.info.off_row_max > 0
    rows, c = int(batch.qo_indptr[-1]), batch.cfg
    out = torch.full((rows, c.num_qo_heads, c.head_dim_vo), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    lse = torch.full((rows, c.num_qo_heads), float("nan"), device="cuda")
    N.nvfp4kv_decode_run_static(plan, g.q, g.cache, g.kv_indices, batch.sm_scale, out=out,
                                lse=lse)
    torch.cuda.synchronize()
    assert N.nvfp4kv_static_workspace_flags(plan) == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
