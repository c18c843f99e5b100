"""Page size 1 and f16 output on the GPU, against the float64 oracle.

Page size 1 (page "Re-enable split-KV for NVFP4 KV cache in prefill path":
the asymmetric NVFP4 paged-prefill tests run page sizes 1 and 16): every
token has its own page, in a random permutation of the pool; the kernels
gather a tile's 16 token rows from 16 pages.  The quantiser must stay
byte-identical, attention within the usual tolerances, on the tiny, batched
and asymmetric-head decode shapes, causal extend on the tcgen05 kernel, the
CUDA-core kernel, split and unsplit plans, NHD and HND caches, the fused
append and the page-order invariance with a poisoned pool.

f16 output (a configurable output dtype, as in the optimisation pull
request inlined in page "fix(attention): correct SM120 NVFP4 qk_correction
layout, row-sum reduction, and lse"): the same results rounded to f16, within
5e-3 beyond f16's half ulp, on every kernel family and both merges."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle as O
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def small(page_size=1, extra_pages=0, **kw):
    args = dict(seed=51, kv_lens=(1, 16, 17, 33, 250, 1000), qo_len=1, num_qo_heads=8,
                num_kv_heads=2, head_dim_qk=128, head_dim_vo=128)
    args.update(kw)
    args["batch"] = len(args["kv_lens"])
    b = W.make_batch(W.custom_workload(**args))
    return W.with_page_size_one(b, extra_pages=extra_pages) if page_size == 1 else b


def check(batch, layout="HND", **plan_kw):
    g = H.GpuCase(batch, layout=layout, **plan_kw)
    assert int(g.flags.item()) == 0
    oc, pt = H.oracle_cache(batch, layout)
    H.compare_cache_bytes(g.cache, oc)
    out, lse = g.run()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    ro, rl = H.oracle_attention(batch, oc, pt)
    return H.compare(out, lse, ro, rl), g


@pytest.mark.parametrize("name", ["tiny_decode", "batched_decode", "asymmetric_heads_decode"])
def test_page_size_one_workloads(name):
    batch = W.with_page_size_one(W.make_batch(W.WORKLOADS[name]))
    stats, g = check(batch)
    assert g.plan.info.page_size == 1
    print(name, stats)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("kw", [dict(disable_split=True), dict(force_chunk_tokens=32),
                                dict(force_chunk_tokens=256)])
def test_page_size_one_split_and_layouts(layout, kw):
    check(small(), layout, **kw)


@pytest.mark.parametrize("dk,dv", [(64, 64), (256, 128), (512, 256)])
def test_page_size_one_head_dims(dk, dv):
    check(small(head_dim_qk=dk, head_dim_vo=dv, kv_lens=(5, 40, 300)), force_chunk_tokens=64)


@pytest.mark.parametrize("kernel,qo_len", [(1, 4), (2, 1), (2, 4), (3, 16), (3, 1)])
def test_page_size_one_kernels(kernel, qo_len):
    batch = small(qo_len=qo_len, causal=qo_len > 1, kv_lens=(16, 40, 161, 700))
    stats, g = check(batch, kernel=kernel, force_chunk_tokens=128)
    assert g.plan.info.kernel == kernel


def test_page_size_one_fused_append():
    batch = small(kv_lens=(16, 17, 40, 161, 700), qo_len=4, causal=True)
    g = H.GpuCase(batch, append=False, force_chunk_tokens=64)
    g.append(batch.prefix)
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) + batch.new.positions.long())
    out, lse = N.nvfp4kv_decode_append_run(g.plan, batch.new.k[order].cuda(),
                                           batch.new.v[order].cuda(), g.q, g.cache,
                                           g.kv_indices, batch.sm_scale)
    torch.cuda.synchronize()
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    oc, pt = H.oracle_cache(batch)
    H.compare_cache_bytes(g.cache, oc)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


def test_page_size_one_prefix_cache_extend_sample():
    """The prefix-cache extend workload over 1-token pages (shared prefix
    tokens in shared pages), tcgen05 kernel, checked on three requests."""
    batch = W.with_page_size_one(W.make_batch(W.WORKLOADS["prefix_cache_extend"]))
    order = np.argsort(batch.kv_lens)
    requests = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    g = H.GpuCase(batch)
    assert g.plan.info.kernel == 3
    oc, pt = H.oracle_cache(batch, requests=requests)
    out, lse = g.run()
    ro, rl = H.oracle_attention(batch, oc, pt, requests)
    H.compare(out, lse, ro, rl)
    assert bool(torch.isfinite(out.float()).all())


def test_page_size_one_poisoned_pool_and_permutation():
    base = small(page_size=16, kv_lens=(37, 100, 260))
    b1 = W.with_page_size_one(base, extra_pages=11)
    g1 = H.GpuCase(b1, fill=0xFF, force_chunk_tokens=48)
    o1, l1 = g1.run()
    b2 = W.with_page_size_one(base, seed=99, extra_pages=11)
    g2 = H.GpuCase(b2, fill=0xFF, force_chunk_tokens=48)
    o2, l2 = g2.run()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    assert not torch.isnan(o1.float()).any()


def test_page_size_one_dequantize_bit_exact():
    batch = small(kv_lens=(17, 40))
    g = H.GpuCase(batch)
    oc, _ = H.oracle_cache(batch)
    k, v = N.nvfp4kv_dequantize_paged(g.cache, g.kv_indices, device_flags=g.flags)
    torch.cuda.synchronize()
    assert k.shape[1] == 1 and int(g.flags.item()) == 0
    k, v = k.cpu().numpy(), v.cpu().numpy()
    for e, page in enumerate(g.kv_indices.cpu().tolist()):
        for h in range(batch.cfg.num_kv_heads):
            rk = O.dequant_row(oc, 0, page, 0, h).astype(np.float32)
            rv = O.dequant_row(oc, 1, page, 0, h).astype(np.float32)
            assert np.array_equal(k[e, 0, h].view(np.uint32), rk.view(np.uint32))
            assert np.array_equal(v[e, 0, h].view(np.uint32), rv.view(np.uint32))


# ---- f16 output ------------------------------------------------------------

@pytest.mark.parametrize("kernel,layout,qo_len,kw", [
    (1, "HND", 1, dict(force_chunk_tokens=64)),      # the decode kernel, split merge
    (1, "HND", 1, dict(disable_split=True)),
    (1, "NHD", 4, dict(force_chunk_tokens=64)),      # the register kernel
    (2, "HND", 1, dict(force_chunk_tokens=64)),      # CUDA cores
    (3, "HND", 16, dict(force_chunk_tokens=128))])   # tcgen05
def test_f16_output(kernel, layout, qo_len, kw):
    batch = small(page_size=16, qo_len=qo_len, causal=qo_len > 1, kv_lens=(16, 40, 161, 700))
    stats, g = check(batch, layout, kernel=kernel, out_dtype=torch.float16, **kw)
    out, _ = g.run()
    assert out.dtype == torch.float16
    # the bf16 plan's output agrees with the f16 one to bf16 rounding
    c = batch.cfg
    pb = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                               c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                               causal=c.causal, kernel=kernel, **kw)
    ob, _ = g.run(pb)
    assert torch.equal(out.float().to(torch.bfloat16).view(torch.int16), ob.view(torch.int16)) \
        or float((out.float() - ob.float()).abs().max()) <= 2 ** -7 * float(ob.float().abs().max())


def test_f16_output_standalone_merge():
    batch = small(page_size=16, kv_lens=(100, 1000, 3000))
    g = H.GpuCase(batch, force_chunk_tokens=64, out_dtype=torch.float16)
    out, lse = g.run()
    out2, lse2 = out.clone(), lse.clone()
    N.nvfp4kv_decode_merge(g.plan, out2, lse2)
    torch.cuda.synchronize()
    a, b = out.float(), out2.float()
    ulp = 2.0 ** (torch.floor(torch.log2(torch.clamp(b.abs(), min=2 ** -14))) - 10)
    assert bool(((a - b).abs() <= ulp).all())
    assert float((lse - lse2).abs().max()) <= 1e-5
