"""Kernel 4, FP4 query and probabilities, against the float64 oracle of the
same method (orc_attention_unit_fp4qp).

The query is quantised to NVFP4 per 16 dims; a first launch writes each
unit's row maxima and the attention launch quantises p * 2688 against the
row's maximum over all its keys per 16 keys.  The kernel's p is an f32
exponential of f32 scores, the oracle's a float64 one: the FP4 codes agree
unless a value lies within that rounding of a decision boundary, which
these seeded cases do not meet, so the outputs are held to the same bf16
bound as the other kernels."""
import json
import os

import pytest
import torch

import gpu_harness as H
import nvfp4_paged_kv_nvfp4kv_gb300 as N
import oracle as O
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def fp4qp_oracle(batch, layout="HND"):
    oc, pt = H.oracle_cache(batch, layout)
    c = batch.cfg
    return O.attention_fp4qp(oc, pt, batch.qo_indptr, batch.q, c.num_qo_heads, c.causal,
                             batch.sm_scale), oc


def record(name, stats):
    path = os.environ.get("NVFP4KV_FP4QP_STATS")
    if path:
        d = json.load(open(path)) if os.path.exists(path) else {}
        d[name] = stats
        json.dump(d, open(path, "w"), indent=1)


@pytest.mark.parametrize("kv_lens,qo_len,hq,hkv,dk,layout,chunk,causal", [
    ((37, 100, 700), 1, 8, 1, 128, "HND", 0, False),
    ((37, 100, 700), 1, 8, 2, 128, "NHD", 0, False),
    ((16, 2000, 4100), 1, 4, 1, 128, "HND", 512, False),   # split + merge
    ((33, 517), 2, 8, 2, 64, "HND", 0, True),              # 2 positions x G = 4
    ((16, 2000, 4100), 2, 8, 2, 64, "NHD", 1024, True),     # both
])
def test_fp4qp_matches_oracle(kv_lens, qo_len, hq, hkv, dk, layout, chunk, causal):
    cfg = W.custom_workload(seed=41, batch=len(kv_lens), kv_lens=kv_lens, qo_len=qo_len,
                            num_qo_heads=hq, num_kv_heads=hkv, head_dim_qk=dk, head_dim_vo=dk,
                            causal=causal)
    batch = W.make_batch(cfg)
    g = H.GpuCase(batch, layout=layout, kernel=4, force_chunk_tokens=chunk)
    assert g.plan.info.kernel == 4
    if chunk:
        assert g.plan.info.split and g.plan.info.chunk_pages == chunk // 16
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    (ro, rl), _ = fp4qp_oracle(batch, layout)
    stats = H.compare(out, lse, ro, rl)
    record("%s-%d-%d-%d-%s-%d-%d" % (len(kv_lens), qo_len, hq, dk, layout, chunk, causal), stats)


def test_fp4qp_fused_append():
    """The fused append runs in the row-maximum launch: cache bytes equal the
    oracle's, and the attention launch reads the stored tokens."""
    cfg = W.custom_workload(seed=43, batch=3, kv_lens=(40, 333, 1500), qo_len=1,
                            num_qo_heads=8, num_kv_heads=1)
    batch = W.make_batch(cfg)
    g = H.GpuCase(batch, append=False, kernel=4)
    g.append(batch.prefix)
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) + batch.new.positions.long())
    nk, nv = batch.new.k[order].cuda(), batch.new.v[order].cuda()
    out, lse = N.nvfp4kv_decode_append_run(g.plan, nk, nv, g.q, g.cache, g.kv_indices,
                                           batch.sm_scale)
    torch.cuda.synchronize()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    (ro, rl), oc = fp4qp_oracle(batch)
    H.compare_cache_bytes(g.cache, oc)
    record("fused_append", H.compare(out, lse, ro, rl))


def test_fp4qp_page_size_one_and_f16_out():
    """1-token pages in a permuted pool (a 16-key block of P spans 16 pages)
    with f16 outputs and 256-token chunks."""
    base = W.make_batch(W.custom_workload(seed=47, batch=3, kv_lens=(37, 300, 1500), qo_len=1,
                                          num_qo_heads=8, num_kv_heads=1))
    batch = W.with_page_size_one(base)
    g = H.GpuCase(batch, kernel=4, out_dtype=torch.float16, force_chunk_tokens=256)
    assert g.plan.info.kernel == 4 and g.plan.info.split and g.plan.info.page_size == 1
    out, lse = g.run()
    assert out.dtype == torch.float16
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    (ro, rl), _ = fp4qp_oracle(batch)
    record("page_size_one_f16", H.compare(out, lse, ro, rl))


def test_fp4qp_live_lengths():
    """A plan with live last-page lengths: both launches read the current
    lengths (the row maxima and the attention agree on the keys)."""
    import test_gpu_live_length as LL
    full = (22, 40, 105, 250, 1000, 3000)
    cut = [L - 5 for L in full]
    batch = LL.batch_of(full, qo_len=1)
    g = H.GpuCase(batch, append=False)
    g.append(LL.tokens_below(batch, full))
    c = batch.cfg
    np_ = (batch.kv_indptr[1:] - batch.kv_indptr[:-1]).tolist()
    live = H.dev_i32([L - (n - 1) * 16 for L, n in zip(cut, np_)])
    plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 kernel=4, force_chunk_tokens=128, device_last_page_len=live)
    assert plan.info.kernel == 4 and plan.info.split == 1
    out, lse = g.run(plan)
    assert N.nvfp4kv_workspace_flags(plan) == 0
    oc, pt = LL.oracle_at(batch, cut)
    ro, rl = O.attention_fp4qp(oc, pt, batch.qo_indptr, batch.q, c.num_qo_heads, False,
                               batch.sm_scale)
    record("live_lengths", H.compare(out, lse, ro, rl))

