"""GPU parity of the tcgen05 attention kernel (plan option kernel=3: K_hat in
tensor memory, tcgen05.mma products, warp-specialised tile pipeline) against
the float64 oracle: decode and causal extend, 16 / 32 / 64 query rows per CTA,
ragged and tiny lengths, split and unsplit, HND and NHD caches, the fused
append, and the full-size head-dim-128 workloads."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from nvfp4_paged_kv_nvfp4kv_gb300 import api as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def small(**kw):
    args = dict(seed=31, kv_lens=(1, 16, 17, 129, 300, 1000), qo_len=1, num_qo_heads=8,
                num_kv_heads=2, head_dim_qk=128, head_dim_vo=128)
    args.update(kw)
    args["batch"] = len(args["kv_lens"])
    return W.make_batch(W.custom_workload(**args))


def check(batch, layout="HND", **plan_kw):
    g = H.GpuCase(batch, layout=layout, kernel=3, **plan_kw)
    assert g.plan.info.kernel == 3
    oc, pt = H.oracle_cache(batch, layout)
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    ro, rl = H.oracle_attention(batch, oc, pt)
    return H.compare(out, lse, ro, rl), g, (out, lse)


def test_tcgen05_tiny_decode():
    batch = small(kv_lens=(37, 100))
    stats, g, _ = check(batch, disable_split=True)
    assert g.plan.info.rows_per_block == 16


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("split", ["none", "tile", "two_tiles"])
@pytest.mark.parametrize("qo_len,causal,rows", [(1, False, 16), (4, True, 16), (7, True, 32),
                                                (16, True, 64)])
def test_tcgen05_shapes(layout, split, qo_len, causal, rows):
    batch = small(qo_len=qo_len, causal=causal,
                  kv_lens=(16, 17, 129, 300, 1000) if qo_len > 1 else (1, 16, 17, 129, 300, 1000))
    kw = {"none": dict(disable_split=True), "tile": dict(force_chunk_tokens=128),
          "two_tiles": dict(force_chunk_tokens=256)}[split]
    stats, g, _ = check(batch, layout=layout, **kw)
    assert g.plan.info.rows_per_block == rows
    if split != "none":
        assert g.plan.info.split == 1


def test_tcgen05_more_rows_than_a_block():
    # G * n = 4 * 20 = 80 rows: two row blocks of 64
    batch = small(qo_len=20, causal=True, kv_lens=(20, 150, 700))
    stats, g, _ = check(batch, force_chunk_tokens=256)
    assert g.plan.info.row_blocks == 2


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (32, 4)])
def test_tcgen05_group_sizes(hq, hkv):
    batch = small(num_qo_heads=hq, num_kv_heads=hkv, kv_lens=(33, 513))
    check(batch)


def test_tcgen05_agrees_with_mma_sync():
    batch = small(qo_len=3, causal=True, kv_lens=(40, 333, 2000))
    _, _, (o3, l3) = check(batch)
    g1 = H.GpuCase(batch, kernel=1)
    o1, l1 = g1.run()
    assert float((o3.float() - o1.float()).abs().max()) <= 1e-2
    assert float((l3 - l1).abs().max()) <= 2e-3


@pytest.mark.parametrize("qo_len,causal", [(1, False), (16, True)])
def test_tcgen05_fused_append(qo_len, causal):
    batch = small(kv_lens=(16, 17, 40, 161, 700), qo_len=qo_len, causal=causal)
    g = H.GpuCase(batch, append=False, kernel=3, force_chunk_tokens=128)
    g.append(batch.prefix)
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) + batch.new.positions.long())
    out, lse = N.nvfp4kv_decode_append_run(g.plan, batch.new.k[order].cuda(),
                                           batch.new.v[order].cuda(), g.q, g.cache,
                                           g.kv_indices, batch.sm_scale)
    torch.cuda.synchronize()
    oc, pt = H.oracle_cache(batch)
    H.compare_cache_bytes(g.cache, oc)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


@pytest.mark.parametrize("name", ["batched_decode", "long_context_decode",
                                  "prefix_cache_extend"])
def test_tcgen05_workloads(name):
    batch = W.make_batch(W.WORKLOADS[name])
    requests = None
    if name == "prefix_cache_extend":
        order = np.argsort(batch.kv_lens)
        requests = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    g = H.GpuCase(batch, kernel=3)
    oc, pt = H.oracle_cache(batch, requests=requests)
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    ro, rl = H.oracle_attention(batch, oc, pt, requests)
    H.compare(out, lse, ro, rl)


def test_tcgen05_page_order_invariance_with_poison():
    """Pool bytes 0xFF everywhere outside the written slots (NaN scales in
    the tail slots and unused pages): results are bit-identical under a
    permutation of the physical pages, and finite."""
    batch = small(qo_len=16, causal=True, kv_lens=(37, 300, 1000))
    b1 = W.make_batch(batch.cfg, extra_pages=9)
    g1 = H.GpuCase(b1, fill=0xFF, kernel=3, force_chunk_tokens=256)
    o1, l1 = g1.run()
    perm = torch.randperm(b1.num_pages, generator=torch.Generator().manual_seed(5))
    b1.kv_indices = perm[b1.kv_indices.long()].to(torch.int32)
    g2 = H.GpuCase(b1, fill=0xFF, kernel=3, force_chunk_tokens=256)
    o2, l2 = g2.run()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    assert not torch.isnan(o1.float()).any()


def test_tcgen05_bad_page_index_sets_flag_without_fault():
    batch = small(qo_len=16, causal=True, kv_lens=(40, 300))
    g = H.GpuCase(batch, kernel=3)
    assert N.nvfp4kv_workspace_flags(g.plan, clear=True) == 0
    bad = g.kv_indices.clone()
    bad[3] = batch.num_pages + 5
    rows = int(batch.qo_indptr[-1])
    out = torch.empty((rows, 8, 128), dtype=torch.bfloat16, device="cuda")
    N.nvfp4kv_decode_run(g.plan, g.q, g.cache, bad, batch.sm_scale, out=out)
    torch.cuda.synchronize()
    assert N.nvfp4kv_workspace_flags(g.plan, clear=True) & 0x1
    out2, _ = g.run()  # the context still works and the good table is clean
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    assert not torch.isnan(out2.float()).any()


def test_tcgen05_causal_rows_that_start_late_in_a_split():
    """Short chunks over the new tokens: in the last units some query rows
    see no token of the first tile (their maximum is set on a later tile)."""
    batch = small(qo_len=16, causal=True, kv_lens=(16, 140, 395))
    check(batch, force_chunk_tokens=128)
    check(batch, force_chunk_tokens=256)


def test_tcgen05_v_ones_and_q_zero_probes():
    batch = small(qo_len=16, causal=True, kv_lens=(37, 100, 250))
    for ts in (batch.prefix, batch.new):
        ts.v.fill_(1.0)
    batch.q.zero_()
    g = H.GpuCase(batch, kernel=3, force_chunk_tokens=128)
    out, lse = g.run()
    assert torch.all(out.float() == 1.03125)
    # uniform scores: lse = ln(number of visible keys) for every row
    import math
    want = []
    for b, L in enumerate(batch.kv_lens):
        for i in range(16):
            want.append([math.log(L - 16 + i + 1)] * 8)
    want = torch.tensor(want, device="cuda", dtype=torch.float32)
    assert torch.allclose(lse, want, atol=1e-5, rtol=0)
