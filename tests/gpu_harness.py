"""Shared helpers of the GPU tests: run the CUDA path through the C ABI on a
seeded Batch, run the float64 oracle on the same bf16 inputs (never on
anything the GPU produced), and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

OUT_ATOL = 5e-3   # max-abs on bf16 outputs vs the float64 oracle
LSE_ATOL = 1e-3   # max-abs on lse


def dev_i32(t):
    return torch.as_tensor(t).to(torch.int32).cuda()


class GpuCase:
    """Cache filled by the GPU quantiser, a plan, and one run."""

    def __init__(self, batch: W.Batch, layout="HND", pad_page_bytes=0, fill=0,
                 append=True, **plan_kw):
        self.batch = batch
        c = batch.cfg
        self.layout = batch.cache_layout(layout, pad_page_bytes)
        self.cache = N.PagedCache.allocate(self.layout, batch.k_global_scale,
                                           batch.v_global_scale, fill=fill)
        self.kv_indices = dev_i32(batch.kv_indices)
        self.kv_indptr = dev_i32(batch.kv_indptr)
        self.last = dev_i32(batch.last_page_len)
        self.q = batch.q.cuda()
        self.flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        if append:
            self.append(batch.prefix)
            self.append(batch.new)
        plan_kw.setdefault("page_size", batch.page_size)
        self.plan = N.nvfp4kv_decode_plan(
            batch.qo_indptr, batch.kv_indptr, batch.last_page_len, c.num_qo_heads,
            c.num_kv_heads, c.head_dim_qk, c.head_dim_vo, causal=c.causal, **plan_kw)

    def append(self, ts, chunk=65536):
        n = ts.k.shape[0]
        for s in range(0, n, chunk):
            N.nvfp4kv_quantize_append(
                self.cache, ts.k[s:s + chunk].cuda(), ts.v[s:s + chunk].cuda(),
                dev_i32(ts.batch_idx[s:s + chunk]), dev_i32(ts.positions[s:s + chunk]),
                self.kv_indices, self.kv_indptr, self.last, device_flags=self.flags)
        torch.cuda.synchronize()

    def run(self, plan=None, q=None):
        plan = plan or self.plan
        c = self.batch.cfg
        rows = int(self.batch.qo_indptr[-1])
        dt = torch.float16 if plan.info.out_dtype == 1 else torch.bfloat16
        out = torch.full((rows, c.num_qo_heads, c.head_dim_vo), float("nan"),
                         dtype=dt, device="cuda")
        lse = torch.full((rows, c.num_qo_heads), float("nan"), device="cuda")
        N.nvfp4kv_decode_run(plan, self.q if q is None else q, self.cache, self.kv_indices,
                             self.batch.sm_scale, out=out, lse=lse)
        torch.cuda.synchronize()
        return out, lse


def token_subset(ts: W.TokenSet, mask) -> W.TokenSet:
    return W.TokenSet(ts.batch_idx[mask], ts.positions[mask], ts.k[mask], ts.v[mask])


def oracle_cache(batch: W.Batch, layout="HND", requests=None, pad_page_bytes=0, fill=0):
    """Oracle-quantised cache, of every token or only of the tokens the given
    requests can see (their own tokens and the shared prefix)."""
    if requests is None:
        return O.cache_from_batch(batch, layout, fill, pad_page_bytes)
    c = O.Cache(batch.cache_layout(layout, pad_page_bytes), batch.k_global_scale,
                batch.v_global_scale, fill)
    pt = O.PageTable.of(batch)
    req = torch.tensor(sorted(requests))
    S = batch.cfg.shared_prefix_tokens
    for ts in (batch.prefix, batch.new):
        m = torch.isin(ts.batch_idx, req.to(ts.batch_idx.dtype))
        if S:
            m |= (ts.batch_idx == 0) & (ts.positions < S)
        rc = O.quantize_append(c, pt, token_subset(ts, m))
        assert rc == 0
    return c, pt


def oracle_attention(batch: W.Batch, cache, pt, requests=None, chunk_tokens=0):
    c = batch.cfg
    units = None
    if requests is not None:
        units = [(b, h) for b in requests for h in range(c.num_kv_heads)]
    return O.attention(cache, pt, batch.qo_indptr, batch.q, c.num_qo_heads, c.causal,
                       batch.sm_scale, units=units, chunk_tokens=chunk_tokens)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def bf16_half_ulp(x: np.ndarray, mant_bits: int = 7) -> np.ndarray:
    """Half an ulp at |x| of a format with mant_bits stored mantissa bits
    (7: bf16, 10: f16)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(a)) - mant_bits)


def compare(out_gpu, lse_gpu, out_orc, lse_orc, atol=OUT_ATOL, lse_atol=LSE_ATOL):
    """Element-wise comparison on the rows the oracle computed.

    The output is bf16, so even an exact result differs from the float64
    oracle by up to half a bf16 ulp (0.0078 once |o| >= 2); the 5e-3 budget
    is applied to the arithmetic on top of that rounding:
    |gpu - oracle| <= 5e-3 + ulp_bf16(max(|gpu|, |oracle|)) / 2,
    and plainly |gpu - oracle| <= 5e-3 where both are below 1 in magnitude.
    Returns the error statistics; asserts the tolerances and no NaN."""
    og = out_gpu.float().cpu().double().numpy()
    lg = lse_gpu.cpu().double().numpy()
    sel = ~np.isnan(lse_orc)
    assert sel.any()
    assert not np.isnan(og[sel]).any(), "NaN in GPU output"
    assert not np.isnan(lg[sel]).any(), "NaN in GPU lse"
    d = np.abs(og[sel] - out_orc[sel])
    dl = np.abs(lg[sel] - lse_orc[sel])
    mant = 10 if out_gpu.dtype == torch.float16 else 7
    excess = d - bf16_half_ulp(np.maximum(np.abs(og[sel]), np.abs(out_orc[sel])), mant)
    ref = out_orc[sel].reshape(-1)
    got = og[sel].reshape(-1)
    stats = {
        "max_abs": float(d.max()),
        "max_abs_beyond_bf16_rounding": float(excess.max()),
        "max_abs_vs_bf16_oracle": float(np.abs(og[sel] - bf16_round(out_orc[sel])).max()),
        "lse_max_abs": float(dl.max()),
        "alpha": float(np.dot(got, ref) / np.dot(ref, ref)) if np.dot(ref, ref) > 0 else 1.0,
        "nan": int(np.isnan(og).sum()),
    }
    # where |o| < 1 the bf16 half-ulp is at most 2^-9, and the plain 5e-3
    # bound holds by itself
    small = np.maximum(np.abs(og[sel]), np.abs(out_orc[sel])) < 1.0
    stats["max_abs_where_below_1"] = float(d[small].max()) if small.any() else 0.0
    assert stats["max_abs_beyond_bf16_rounding"] <= atol, stats
    assert stats["max_abs_where_below_1"] <= atol, stats
    assert stats["lse_max_abs"] <= lse_atol, stats
    return stats


def compare_cache_bytes(gcache: N.PagedCache, ocache: O.Cache, pages=None):
    """Byte equality of the four buffers (optionally only the given pages)."""
    lay = ocache.layout
    rows = lay.rows()
    for w in ("k_data", "v_data", "k_sf", "v_sf"):
        g = getattr(gcache, w).cpu().numpy()
        o = ocache.bufs[w]
        if pages is None:
            bad = np.nonzero(g != o)[0]
            assert bad.size == 0, "%s differs at %d bytes, first %r" % (w, bad.size, bad[:8])
        else:
            sp = lay.strides(rows[w])[0]
            for p in pages:
                a, b = p * sp, (p + 1) * sp
                assert np.array_equal(g[a:b], o[a:b]), "%s differs in page %d" % (w, p)
