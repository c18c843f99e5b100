"""Plans with live last-page lengths (plan option device_last_page_len): the
kernels read each request's current last_page_len from a device array, so
one plan serves successive decode steps while page and query counts hold.

Checked against the float64 oracle at the current lengths: a plan made with
stale lengths on every kernel family, a three-step decode loop with the
fused append and one plan, and the flag for a bad live length."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle as O
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import _lib
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def batch_of(kv_lens, qo_len=1, hq=8, hkv=2, causal=False, seed=41, dk=128, dv=128):
    cfg = W.custom_workload(seed=seed, batch=len(kv_lens), kv_lens=kv_lens, qo_len=qo_len,
                            num_qo_heads=hq, num_kv_heads=hkv, causal=causal,
                            head_dim_qk=dk, head_dim_vo=dv)
    return W.make_batch(cfg)


def tokens_below(batch, lens):
    """The batch's tokens at positions below lens[b] (all tokens, prefix and
    new, regrouped)."""
    ts = [batch.prefix, batch.new]
    bi = torch.cat([t.batch_idx for t in ts])
    pos = torch.cat([t.positions for t in ts])
    k = torch.cat([t.k for t in ts])
    v = torch.cat([t.v for t in ts])
    lim = torch.tensor(lens, dtype=torch.int32)[bi.long()]
    m = pos < lim
    return W.TokenSet(bi[m], pos[m], k[m], v[m])


def oracle_at(batch, lens, layout="HND"):
    """Oracle cache and page table for the requests cut to lengths `lens`
    (same pages)."""
    c = O.Cache(batch.cache_layout(layout), batch.k_global_scale, batch.v_global_scale)
    np_ = (batch.kv_indptr[1:] - batch.kv_indptr[:-1]).tolist()
    lpl = [L - (n - 1) * 16 for L, n in zip(lens, np_)]
    pt = O.PageTable(batch.kv_indices, batch.kv_indptr, torch.tensor(lpl, dtype=torch.int32))
    assert O.quantize_append(c, pt, tokens_below(batch, lens)) == 0
    return c, pt


@pytest.mark.parametrize("kernel,layout,qo_len,causal", [
    (1, "HND", 1, False), (1, "NHD", 1, False), (1, "HND", 4, True), (2, "HND", 1, False),
    (3, "HND", 16, True)])
def test_stale_plan_reads_current_lengths(kernel, layout, qo_len, causal):
    # full lengths keep every request's page count when cut by up to 5 tokens
    full = (22, 40, 105, 250, 1000, 3000)
    batch = batch_of(full, qo_len=qo_len, causal=causal)
    cut = [L - 5 for L in full]
    assert all(L - 5 > (L - 1) // 16 * 16 for L in full)
    g = H.GpuCase(batch, layout=layout, append=False)
    g.append(tokens_below(batch, full))
    c = batch.cfg
    np_ = (batch.kv_indptr[1:] - batch.kv_indptr[:-1]).tolist()
    live = H.dev_i32([L - (n - 1) * 16 for L, n in zip(cut, np_)])
    plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 causal=causal, kernel=kernel, force_chunk_tokens=128,
                                 device_last_page_len=live)
    assert plan.info.kernel == kernel and plan.info.split == 1
    out, lse = g.run(plan)
    assert N.nvfp4kv_workspace_flags(plan) == 0
    oc, pt = oracle_at(batch, cut, layout)
    ro, rl = O.attention(oc, pt, batch.qo_indptr, batch.q, c.num_qo_heads, causal,
                         batch.sm_scale)
    H.compare(out, lse, ro, rl)


def test_decode_steps_with_one_plan_and_fused_append():
    """Three decode steps: each appends one token per request (fused) and
    attends; the plan is made once and only the device last_page_len moves."""
    start = (17, 40, 100, 250, 1000, 3000)       # lengths before the first step
    final = tuple(L + 3 for L in start)          # same page counts throughout
    batch = batch_of(final)
    c = batch.cfg
    np_ = (batch.kv_indptr[1:] - batch.kv_indptr[:-1]).tolist()
    assert all((L + 1 + 15) // 16 == n for L, n in zip(start, np_))
    g = H.GpuCase(batch, append=False)
    g.append(tokens_below(batch, start))
    live = H.dev_i32([L + 1 - (n - 1) * 16 for L, n in zip(start, np_)])
    plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 force_chunk_tokens=256, device_last_page_len=live)
    allt = tokens_below(batch, final)
    for s in range(3):
        lens = [L + s + 1 for L in start]
        live.copy_(H.dev_i32([L - (n - 1) * 16 for L, n in zip(lens, np_)]))
        # the step's new token of each request, row-aligned with q
        rows = []
        for b in range(c.batch):
            m = (allt.batch_idx == b) & (allt.positions == lens[b] - 1)
            rows.append(int(torch.nonzero(m)[0]))
        nk, nv = allt.k[rows].cuda(), allt.v[rows].cuda()
        out, lse = N.nvfp4kv_decode_append_run(plan, nk, nv, g.q, g.cache, g.kv_indices,
                                               batch.sm_scale)
        torch.cuda.synchronize()
        assert N.nvfp4kv_workspace_flags(plan) == 0
        oc, pt = oracle_at(batch, lens)
        H.compare_cache_bytes(g.cache, oc)
        ro, rl = O.attention(oc, pt, batch.qo_indptr, batch.q, c.num_qo_heads, False,
                             batch.sm_scale)
        H.compare(out, lse, ro, rl)


def test_bad_live_length_sets_flag_without_fault():
    batch = batch_of((40, 100))
    g = H.GpuCase(batch)
    c = batch.cfg
    live = H.dev_i32([0, 17])
    plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 device_last_page_len=live)
    out, _ = g.run(plan)
    assert N.nvfp4kv_workspace_flags(plan, clear=True) & _lib.FLAG_BAD_LIVE_LENGTH
    assert bool(torch.isfinite(out.float()).all())
    live.copy_(batch.last_page_len.to(torch.int32).cuda())
    out2, _ = g.run(plan)
    assert N.nvfp4kv_workspace_flags(plan) == 0
    ref, _ = g.run()
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))
