"""GPU edge cases against the oracle: ragged and tiny lengths, empty query
sets, every head-dim pair and GQA group size, NHD / HND / padded layouts and
independent K/V stride families, page-order invariance with poisoned unused
pages, the pages' uniform-score probes, device-side index checks, and the
standalone merge."""
import math

import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle as O
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def small(**kw):
    args = dict(seed=21, kv_lens=(1, 16, 17, 31, 33, 250), qo_len=1, num_qo_heads=8,
                num_kv_heads=2, head_dim_qk=128, head_dim_vo=128)
    args.update(kw)
    args["batch"] = len(args["kv_lens"])
    return W.make_batch(W.custom_workload(**args))


def check(batch, layout="HND", pad_page_bytes=0, **plan_kw):
    g = H.GpuCase(batch, layout=layout, pad_page_bytes=pad_page_bytes, **plan_kw)
    oc, pt = H.oracle_cache(batch, layout, pad_page_bytes=pad_page_bytes)
    H.compare_cache_bytes(g.cache, oc)
    out, lse = g.run()
    ro, rl = H.oracle_attention(batch, oc, pt)
    return H.compare(out, lse, ro, rl), g, (out, lse)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("split", [False, True])
def test_ragged_lengths(layout, split):
    kw = dict(force_chunk_tokens=32) if split else dict(disable_split=True)
    check(small(), layout, **kw)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (256, 256), (256, 128), (512, 256)])
def test_head_dims(dk, dv):
    check(small(head_dim_qk=dk, head_dim_vo=dv, kv_lens=(5, 40, 300)), force_chunk_tokens=64)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 1), (16, 2), (32, 1), (12, 4)])
def test_group_sizes(hq, hkv):
    check(small(num_qo_heads=hq, num_kv_heads=hkv, kv_lens=(3, 77, 129)))


@pytest.mark.parametrize("qo_len", [2, 5, 16])
def test_causal_extend(qo_len):
    check(small(qo_len=qo_len, causal=True, kv_lens=(16, 40, 161)), force_chunk_tokens=32)


def test_extend_all_tokens_new_and_shared_prefix():
    batch = small(qo_len=16, causal=True, kv_lens=(16, 80, 1100, 2000),
                  shared_prefix_tokens=0)
    check(batch)
    batch2 = small(qo_len=8, causal=True, kv_lens=(1030, 1100, 1500), shared_prefix_tokens=1024)
    check(batch2)


def test_requests_without_queries():
    batch = small(kv_lens=(20, 50, 70, 90), qo_len=2, causal=True)
    # requests 0 and 2 ask no query rows; 1 and 3 keep theirs
    keep = torch.tensor([2, 3, 6, 7])
    batch.q = batch.q[keep].contiguous()
    batch.qo_indptr = torch.tensor([0, 0, 2, 2, 4], dtype=torch.int32)
    check(batch)
    check(batch, force_chunk_tokens=16)


def test_padded_pages_and_independent_kv_strides():
    batch = small(kv_lens=(37, 100, 260))
    check(batch, "HND", pad_page_bytes=48)
    # K pool HND, V pool NHD with padding: separate stride families
    g = H.GpuCase(batch, append=False)
    lay_v = batch.cache_layout("NHD", pad_page_bytes=96)
    for w in ("v_data", "v_sf"):
        n = lay_v.nbytes(w)
        setattr(g.cache, w, torch.zeros(n, dtype=torch.uint8, device="cuda"))
        g.cache.strides[w] = lay_v.strides(lay_v.rows()[w])
    g.append(batch.prefix)
    g.append(batch.new)
    oc, pt = H.oracle_cache(batch, "HND")
    out, lse = g.run()
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


def test_page_order_invariance_with_poison():
    batch = small(kv_lens=(37, 100, 260))
    b1 = W.make_batch(batch.cfg, extra_pages=7)
    g1 = H.GpuCase(b1, fill=0xFF, force_chunk_tokens=48)
    o1, l1 = g1.run()
    perm = torch.randperm(b1.num_pages, generator=torch.Generator().manual_seed(3))
    b1.kv_indices = perm[b1.kv_indices.long()].to(torch.int32)
    g2 = H.GpuCase(b1, fill=0xFF, force_chunk_tokens=48)
    o2, l2 = g2.run()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    assert not torch.isnan(o1.float()).any()


def test_v_ones_probe_exact():
    # uniform-score / V = ones probe (page "fix(attention): correct SM120
    # NVFP4 ... lse"): the output is the dequantised value of 1, 1.03125
    batch = small(kv_lens=(37, 100, 250), qo_len=3, causal=True)
    for ts in (batch.prefix, batch.new):
        ts.v.fill_(1.0)
    g = H.GpuCase(batch)
    out, _ = g.run()
    assert torch.all(out.float() == 1.03125)


def test_q_zero_probe_lse_is_ln_len():
    batch = small(kv_lens=(1, 37, 100, 250))
    batch.q.zero_()
    g = H.GpuCase(batch, force_chunk_tokens=32)
    out, lse = g.run()
    want = torch.tensor([math.log(L) for L in batch.kv_lens], device="cuda")
    assert torch.allclose(lse, want[:, None].expand_as(lse), atol=1e-5, rtol=0)
    oc, pt = H.oracle_cache(batch)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


def test_bad_page_index_sets_flag_without_fault():
    batch = small(kv_lens=(37, 100))
    g = H.GpuCase(batch)
    assert N.nvfp4kv_workspace_flags(g.plan, clear=True) == 0
    bad = g.kv_indices.clone()
    bad[1] = batch.num_pages + 5
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    N.nvfp4kv_decode_run(g.plan, g.q, g.cache, bad, batch.sm_scale, out=out)
    torch.cuda.synchronize()
    assert N.nvfp4kv_workspace_flags(g.plan, clear=True) & 0x1
    out2, _ = g.run()  # the context still works and the good table is clean
    assert N.nvfp4kv_workspace_flags(g.plan) == 0
    assert not torch.isnan(out2.float()).any()


def test_append_out_of_range_sets_flag_and_writes_nothing():
    batch = small(kv_lens=(37, 100))
    g = H.GpuCase(batch, append=False)
    before = g.cache.k_data.clone()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = batch.new.k[:1].cuda()
    v = batch.new.v[:1].cuda()
    for b, pos in ((0, 37), (5, 0), (1, -1)):
        N.nvfp4kv_quantize_append(g.cache, k, v, H.dev_i32([b]), H.dev_i32([pos]),
                                  g.kv_indices, g.kv_indptr, g.last, device_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & 0x2
    assert torch.equal(before, g.cache.k_data)


def test_merge_states_matches_oracle():
    rng = np.random.default_rng(5)
    counts = [1, 2, 3, 17, 40, 1, 5]
    P = sum(counts)
    o = rng.standard_normal((P, 128)).astype(np.float32)
    l = (rng.standard_normal(P) * 4).astype(np.float32)
    l[3:6] = -np.inf                     # entry 2 fully masked
    l[40] = -np.inf                      # one masked partial inside entry 4
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    out, lse = N.nvfp4kv_merge_states(torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda(),
                                      torch.from_numpy(indptr).cuda())
    torch.cuda.synchronize()
    for e in range(len(counts)):
        a, b = indptr[e], indptr[e + 1]
        ro, rl = O.merge_states(o[a:b].astype(np.float64), l[a:b].astype(np.float64))
        if rl == -math.inf:
            assert float(lse[e]) == -math.inf and torch.all(out[e] == 0)
            continue
        assert abs(float(lse[e]) - rl) <= 1e-5
        assert np.abs(out[e].float().cpu().numpy() - ro).max() <= 1e-2 * max(1, np.abs(ro).max())


def test_lse_optional():
    batch = small(kv_lens=(37, 100))
    g = H.GpuCase(batch)
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    N.nvfp4kv_decode_run(g.plan, g.q, g.cache, g.kv_indices, batch.sm_scale, out=out,
                         lse=None)
    torch.cuda.synchronize()
    ref, _ = g.run()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (256, 128), (512, 256)])
@pytest.mark.parametrize("causal,qo_len", [(False, 1), (True, 4)])
def test_cuda_core_kernel(dk, dv, causal, qo_len):
    batch = small(head_dim_qk=dk, head_dim_vo=dv, kv_lens=(5, 40, 300), qo_len=qo_len,
                  causal=causal)
    stats, g, _ = check(batch, kernel=2, force_chunk_tokens=64)
    assert g.plan.info.kernel == 2 and g.plan.info.rows_per_block == 8
    stats2, g2, _ = check(batch, kernel=2, disable_split=True)


@pytest.mark.parametrize("layout,kw", [("HND", dict(force_chunk_tokens=32)),
                                       ("NHD", dict(disable_split=True)),
                                       ("HND", dict(disable_split=True))])
@pytest.mark.parametrize("qo_len,causal", [(1, False), (7, True), (16, True)])
def test_fused_append_small(layout, kw, qo_len, causal):
    batch = small(kv_lens=(16, 17, 40, 161), qo_len=qo_len, causal=causal)
    g = H.GpuCase(batch, layout=layout, append=False, **kw)
    g.append(batch.prefix)
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) + batch.new.positions.long())
    out, lse = N.nvfp4kv_decode_append_run(g.plan, batch.new.k[order].cuda(),
                                           batch.new.v[order].cuda(), g.q, g.cache,
                                           g.kv_indices, batch.sm_scale)
    torch.cuda.synchronize()
    oc, pt = H.oracle_cache(batch, layout)
    H.compare_cache_bytes(g.cache, oc)
    ro, rl = H.oracle_attention(batch, oc, pt)
    H.compare(out, lse, ro, rl)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (512, 256)])
def test_dequantize_paged_bit_exact(layout, dk, dv):
    """nvfp4kv_dequantize_paged: every slot of every listed page equals the
    oracle's exact dequantised value rounded to float32, byte for byte."""
    batch = small(kv_lens=(17, 40, 161), head_dim_qk=dk, head_dim_vo=dv)
    g = H.GpuCase(batch, layout=layout)
    oc, _ = H.oracle_cache(batch, layout)
    ids = g.kv_indices
    k, v = N.nvfp4kv_dequantize_paged(g.cache, ids, device_flags=g.flags)
    torch.cuda.synchronize()
    assert int(g.flags.item()) == 0
    k, v = k.cpu().numpy(), v.cpu().numpy()
    c = batch.cfg
    for e, page in enumerate(ids.cpu().tolist()):
        for slot in range(16):
            for h in range(c.num_kv_heads):
                rk = O.dequant_row(oc, 0, page, slot, h).astype(np.float32)
                rv = O.dequant_row(oc, 1, page, slot, h).astype(np.float32)
                assert np.array_equal(k[e, slot, h].view(np.uint32), rk.view(np.uint32))
                assert np.array_equal(v[e, slot, h].view(np.uint32), rv.view(np.uint32))


def test_dequantize_paged_bad_page_and_partial_outputs():
    batch = small(kv_lens=(40,))
    g = H.GpuCase(batch)
    ids = torch.tensor([int(batch.kv_indices[0]), 10 ** 6, -1], dtype=torch.int32,
                       device="cuda")
    k, v = N.nvfp4kv_dequantize_paged(g.cache, ids, want_v=False, device_flags=g.flags)
    torch.cuda.synchronize()
    assert v is None
    assert int(g.flags.item()) & N._lib.FLAG_BAD_PAGE_INDEX
    assert bool((k[1:] == 0).all())
    assert bool((k[0].abs().sum() > 0))


@pytest.mark.parametrize("kernel", [1, 2])
def test_q_rows_wider_than_f16_range(kernel):
    """Q rows whose dynamic range exceeds f16's (about 40 binades).  The
    tensor-core kernel scales each bf16 Q row by a power of two so its
    largest entry lands near 2^14 and converts it to f16: entries more than
    ~2^-38 below the row maximum become f16 subnormals or zero.  Their share
    of a score is below 2^-30 of it, so the results must stay within the
    usual tolerance of the float64 oracle (which keeps every entry): rows of
    tiny values only (2^-100 and 2^-14 times N(0,1)), a 2^6 outlier beside
    entries of 2^-30, and N(0,1) rows with a quarter of the entries at 2^-24
    and a quarter at 2^-60 of their size (60 binades)."""
    batch = small(kv_lens=(37, 100, 250, 1000), num_qo_heads=8, num_kv_heads=2)
    q = batch.q.float()
    gen = torch.Generator().manual_seed(9)
    rows, heads, d = q.shape
    for r in range(rows):
        for h in range(heads):
            kind = (r * heads + h) % 5
            if kind == 0:                     # every entry tiny
                q[r, h] *= 2.0 ** -100
            elif kind == 1:                   # every entry small
                q[r, h] *= 2.0 ** -14
            elif kind == 2:                   # one outlier, the rest tiny
                q[r, h] *= 2.0 ** -30
                q[r, h, int(torch.randint(0, d, (1,), generator=gen))] = 64.0
            elif kind == 3:                   # N(0,1) with entries 2^-24 and 2^-60
                idx = torch.randperm(d, generator=gen)
                q[r, h, idx[: d // 4]] *= 2.0 ** -24
                q[r, h, idx[d // 4: d // 2]] *= 2.0 ** -60
            # kind 4: untouched N(0,1)
    batch.q = q.to(torch.bfloat16)
    stats, g, (out, lse) = check(batch, kernel=kernel, force_chunk_tokens=64)
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
