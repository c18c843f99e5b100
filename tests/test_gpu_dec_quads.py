"""The decode kernel's two launch shapes against the float64 oracle.

A grid of more units than SMs runs four units per CTA (16 warps), paced in
rounds of pages; the last CTA may hold fewer than four units, and its idle
groups only keep the CTA-wide barrier count.  A grid of at most one unit per
SM runs one unit per CTA.  Both are checked on grids built to land on these
edges, with the fused append, causal rows and a live last-page length."""
import pytest
import torch

import gpu_harness as H
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def batch_of(kv_lens, qo_len=1, hq=8, hkv=1, causal=False, seed=83):
    cfg = W.custom_workload(seed=seed, batch=len(kv_lens), kv_lens=kv_lens, qo_len=qo_len,
                            num_qo_heads=hq, num_kv_heads=hkv, causal=causal)
    return W.make_batch(cfg)


def pages(L):
    return (L + 15) // 16


@pytest.mark.parametrize("kv_lens,qo_len,causal", [
    ((16 * 80 + 5, 16 * 79 + 7), 1, False),   # 161 one-page units: the last CTA holds one
    ((16 * 80 + 5, 16 * 79 + 7), 2, True),    # the same with two causal query rows per head
    ((16 * 76 + 1, 16 * 76 + 16), 1, False),  # 153 and 152 units: both sides of the edge
    ((16 * 76, 16 * 76), 1, False),
])
def test_unit_grids_around_one_per_sm(kv_lens, qo_len, causal):
    batch = batch_of(kv_lens, qo_len=qo_len, causal=causal, hq=8 // qo_len)
    g = H.GpuCase(batch, force_chunk_tokens=16)
    units = sum(pages(L) for L in kv_lens)
    assert g.plan.info.num_units == units and g.plan.info.kernel == 1
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    oc, pt = H.oracle_cache(batch)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


def test_fused_append_in_both_shapes():
    """One decode step with the fused append: units above and below one per
    SM give the same cache bytes and outputs within rounding of each other."""
    batch = batch_of((16 * 80 + 5, 16 * 79 + 7), hq=8)
    res = []
    for chunk in (16, 4096):  # 161 units (four per CTA) / 2 units (one per CTA)
        g = H.GpuCase(batch, append=False, force_chunk_tokens=chunk)
        g.append(batch.prefix)
        # new tokens row-aligned with the query rows
        order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) +
                              batch.new.positions.long())
        nk, nv = batch.new.k[order].cuda(), batch.new.v[order].cuda()
        out, lse = N.nvfp4kv_decode_append_run(g.plan, nk, nv, g.q, g.cache, g.kv_indices,
                                               batch.sm_scale)
        torch.cuda.synchronize()
        assert N.nvfp4kv_workspace_flags(g.plan) == 0
        oc, pt = H.oracle_cache(batch)
        H.compare_cache_bytes(g.cache, oc)
        ro, rl = H.oracle_attention(batch, oc, pt)
        H.compare(out, lse, ro, rl)
        res.append(out.float())
    assert torch.allclose(res[0], res[1], atol=2e-3, rtol=0)
