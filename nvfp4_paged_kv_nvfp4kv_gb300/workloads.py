"""Seeded synthetic workloads for NVFP4 paged-KV decode / extend.

This module only draws random inputs and lays out page tables and buffer
shapes; it contains none of the method's arithmetic (no quantisation, no
attention).  Both the CUDA path and the CPU oracle receive exactly these
inputs.

Recipe (every draw uses a CPU ``torch.Generator`` seeded per workload, in the
order listed):
  1. kv lengths: ``randint(lo, hi + 1)`` per request (fixed lengths skip it);
  2. the page permutation: ``randperm`` of the private pages;
  3. outlier channels (batched decode only): first 4 of ``randperm(Dk)``;
  4. Q, then per request K and V: ``randn(float32)`` (outlier K channels
     multiplied by 10) rounded to bf16.
Page size is 16.  Physical page ids of private pages are a random
permutation; pages shared by every request (prefix-cache extend) are ids
0 .. shared-1 and hold the same tokens for every request.

The five workloads follow the configurations of the headline benchmark:
tiny decode, batched decode, long-context split-KV decode, asymmetric heads
(512/256) and prefix-cache extend.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    qo_len: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_vo: int
    kv_len_lo: int
    kv_len_hi: int
    causal: bool = False
    shared_prefix_tokens: int = 0
    k_outlier_channels: int = 0
    amax_global_scale: bool = False
    fixed_kv_lens: Optional[tuple] = None

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads


WORKLOADS: Dict[str, Workload] = {
    "tiny_decode": Workload(
        "tiny_decode", seed=0, batch=2, qo_len=1, num_qo_heads=4, num_kv_heads=1,
        head_dim_qk=128, head_dim_vo=128, kv_len_lo=37, kv_len_hi=100,
        fixed_kv_lens=(37, 100)),
    "batched_decode": Workload(
        "batched_decode", seed=2, batch=16, qo_len=1, num_qo_heads=32,
        num_kv_heads=8, head_dim_qk=128, head_dim_vo=128, kv_len_lo=512,
        kv_len_hi=4096, k_outlier_channels=4, amax_global_scale=True),
    "long_context_decode": Workload(
        "long_context_decode", seed=3, batch=4, qo_len=1, num_qo_heads=32,
        num_kv_heads=8, head_dim_qk=128, head_dim_vo=128, kv_len_lo=32771,
        kv_len_hi=32771, fixed_kv_lens=(32771,) * 4),
    "asymmetric_heads_decode": Workload(
        "asymmetric_heads_decode", seed=4, batch=8, qo_len=1, num_qo_heads=16,
        num_kv_heads=2, head_dim_qk=512, head_dim_vo=256, kv_len_lo=2048,
        kv_len_hi=8192),
    "prefix_cache_extend": Workload(
        "prefix_cache_extend", seed=5, batch=32, qo_len=16, num_qo_heads=32,
        num_kv_heads=8, head_dim_qk=128, head_dim_vo=128, kv_len_lo=2000,
        kv_len_hi=16000, causal=True, shared_prefix_tokens=1024),
}


def custom_workload(name="custom", seed=1, batch=2, qo_len=1, num_qo_heads=4,
                    num_kv_heads=1, head_dim_qk=128, head_dim_vo=128,
                    kv_lens=(37, 100), causal=False, shared_prefix_tokens=0,
                    k_outlier_channels=0, amax_global_scale=False) -> Workload:
    """A small workload with explicit lengths (edge cases in tests)."""
    return Workload(name, seed, batch, qo_len, num_qo_heads, num_kv_heads,
                    head_dim_qk, head_dim_vo, min(kv_lens), max(kv_lens),
                    causal, shared_prefix_tokens, k_outlier_channels,
                    amax_global_scale, tuple(kv_lens))


@dataclasses.dataclass
class CacheLayout:
    """Byte strides of the four paged buffers (innermost row contiguous).

    ``HND``: [page][head][slot][row];  ``NHD``: [page][slot][head][row].
    Row = Dk/2 packed bytes (K), Dv/2 (V), Dk/16 scale bytes (K), Dv/16 (V).
    """
    layout: str
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_vo: int
    pad_page_bytes: int = 0

    def strides(self, row_bytes: int):
        P, H = self.page_size, self.num_kv_heads
        page = P * H * row_bytes + self.pad_page_bytes
        if self.layout == "HND":
            return page, row_bytes, P * row_bytes          # page, slot, head
        if self.layout == "NHD":
            return page, H * row_bytes, row_bytes
        raise ValueError(self.layout)

    def rows(self):
        return {"k_data": self.head_dim_qk // 2, "v_data": self.head_dim_vo // 2,
                "k_sf": self.head_dim_qk // 16, "v_sf": self.head_dim_vo // 16}

    def nbytes(self, which: str) -> int:
        return self.strides(self.rows()[which])[0] * self.num_pages


@dataclasses.dataclass
class TokenSet:
    """bf16 rows of tokens to store: request id, absolute position, K, V."""
    batch_idx: torch.Tensor      # int32 [n]
    positions: torch.Tensor      # int32 [n]
    k: torch.Tensor              # bf16 [n, Hkv, Dk]
    v: torch.Tensor              # bf16 [n, Hkv, Dv]


@dataclasses.dataclass
class Batch:
    cfg: Workload
    kv_lens: List[int]
    qo_indptr: torch.Tensor      # int32 [B+1]
    kv_indptr: torch.Tensor      # int32 [B+1] (pages)
    kv_indices: torch.Tensor     # int32 [nnz_pages]
    last_page_len: torch.Tensor  # int32 [B]
    num_pages: int
    q: torch.Tensor              # bf16 [sum qo, Hq, Dk]
    prefix: TokenSet             # tokens already in the cache
    new: TokenSet                # tokens appended by the step (the last qo_len)
    k_global_scale: float
    v_global_scale: float
    sm_scale: float
    page_size: int = PAGE_SIZE

    def cache_layout(self, layout="HND", pad_page_bytes=0):
        c = self.cfg
        return CacheLayout(layout, self.num_pages, self.page_size,
                           c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                           pad_page_bytes)


def _bf16_randn(gen, shape, outlier=None):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if outlier is not None:
        x[..., outlier] *= 10.0
    return x.to(torch.bfloat16)


def make_batch(cfg: Workload, extra_pages: int = 0) -> Batch:
    """Draw the seeded inputs of a workload.  ``extra_pages`` reserves unused
    physical pages after the used ones (for poisoning tests)."""
    gen = torch.Generator().manual_seed(cfg.seed)
    B, P = cfg.batch, PAGE_SIZE
    if cfg.fixed_kv_lens is not None:
        lens = [int(x) for x in cfg.fixed_kv_lens]
    else:
        lens = torch.randint(cfg.kv_len_lo, cfg.kv_len_hi + 1, (B,),
                             generator=gen).tolist()
    shared_pages = cfg.shared_prefix_tokens // P
    npages = [math.ceil(L / P) for L in lens]
    n_private = sum(n - shared_pages for n in npages)
    perm = torch.randperm(n_private, generator=gen) + shared_pages
    kv_indptr = [0]
    idx: List[int] = []
    off = 0
    for n in npages:
        idx.extend(range(shared_pages))
        idx.extend(perm[off: off + n - shared_pages].tolist())
        off += n - shared_pages
        kv_indptr.append(len(idx))
    last = [L - (n - 1) * P for L, n in zip(lens, npages)]
    outlier = None
    if cfg.k_outlier_channels:
        outlier = torch.randperm(cfg.head_dim_qk, generator=gen)[: cfg.k_outlier_channels]
    nq = cfg.qo_len
    q = _bf16_randn(gen, (B * nq, cfg.num_qo_heads, cfg.head_dim_qk))
    H, Dk, Dv = cfg.num_kv_heads, cfg.head_dim_qk, cfg.head_dim_vo
    S = cfg.shared_prefix_tokens
    ks, vs, bi, pos = [], [], [], []
    if S:
        ks.append(_bf16_randn(gen, (S, H, Dk), outlier))
        vs.append(_bf16_randn(gen, (S, H, Dv)))
        bi.append(torch.zeros(S, dtype=torch.int32))
        pos.append(torch.arange(S, dtype=torch.int32))
    for b, L in enumerate(lens):
        n = L - S
        ks.append(_bf16_randn(gen, (n, H, Dk), outlier))
        vs.append(_bf16_randn(gen, (n, H, Dv)))
        bi.append(torch.full((n,), b, dtype=torch.int32))
        pos.append(torch.arange(S, L, dtype=torch.int32))
    k_all, v_all = torch.cat(ks), torch.cat(vs)
    b_all, p_all = torch.cat(bi), torch.cat(pos)
    # the step's new tokens: the last qo_len positions of every request
    L_of = torch.tensor(lens, dtype=torch.int32)[b_all.long()]
    is_new = p_all >= (L_of - nq)
    if cfg.amax_global_scale:
        gk = float(k_all.float().abs().max()) / (6.0 * 448.0)
        gv = float(v_all.float().abs().max()) / (6.0 * 448.0)
        gk = float(torch.tensor(gk, dtype=torch.float32))
        gv = float(torch.tensor(gv, dtype=torch.float32))
    else:
        gk = gv = 1.0

    def sel(mask):
        return TokenSet(b_all[mask].contiguous(), p_all[mask].contiguous(),
                        k_all[mask].contiguous(), v_all[mask].contiguous())

    return Batch(
        cfg=cfg, kv_lens=lens,
        qo_indptr=torch.arange(0, B * nq + 1, nq, dtype=torch.int32),
        kv_indptr=torch.tensor(kv_indptr, dtype=torch.int32),
        kv_indices=torch.tensor(idx, dtype=torch.int32),
        last_page_len=torch.tensor(last, dtype=torch.int32),
        num_pages=shared_pages + n_private + extra_pages,
        q=q, prefix=sel(~is_new), new=sel(is_new),
        k_global_scale=gk, v_global_scale=gv,
        sm_scale=1.0 / math.sqrt(Dk))


def with_page_size_one(batch: Batch, seed: int = 7, extra_pages: int = 0) -> Batch:
    """The same batch (tokens, queries, scales) over a page table of 1-token
    pages: every request's tokens get a page each, in a seeded random
    permutation of the physical pages; the shared prefix tokens (if any) keep
    shared pages, ids 0 .. S-1, first in every request's list."""
    S = batch.cfg.shared_prefix_tokens
    lens = [int(x) for x in batch.kv_lens]
    n_private = sum(L - S for L in lens)
    gen = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_private, generator=gen) + S
    idx, indptr, off = [], [0], 0
    for L in lens:
        idx.extend(range(S))
        idx.extend(perm[off: off + L - S].tolist())
        off += L - S
        indptr.append(len(idx))
    return dataclasses.replace(
        batch, kv_indptr=torch.tensor(indptr, dtype=torch.int32),
        kv_indices=torch.tensor(idx, dtype=torch.int32),
        last_page_len=torch.ones(len(lens), dtype=torch.int32),
        num_pages=S + n_private + extra_pages, page_size=1)
