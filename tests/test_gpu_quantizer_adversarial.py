"""Adversarial inputs for the bit-exact GPU quantiser.

The corner-case blocks of ``quant_corners`` (element ties at every e2m1
midpoint, amax at and around every E4M3 midpoint times 6 g, saturation, the
scale's underflow edge, signed zeros) with global scales g in
{2^-60, 1/2688, 1, 2^60} are sent through nvfp4kv_quantize_append and
through the fused append of nvfp4kv_decode_append_run (mma.sync and tcgen05
kernels).  The cache bytes must equal the float64 oracle's byte for byte
(page "Support NVFP4 KV cache decode on SM120": packed e2m1 plus per-16 E4M3
scale caches; the exact recipe is the plain reading the oracle writes out)."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle as O
import nvfp4_paged_kv_nvfp4kv_gb300 as N
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W
from quant_corners import GLOBAL_SCALES, adversarial_blocks, bf16

pytestmark = pytest.mark.gpu


def adversarial_batch(g: float, seed: int, hkv=2, hq=4, d=128):
    """A batch whose requests hold only new tokens (kv_len = qo_len = 16,
    causal), with K and V rows made of the corner-case blocks."""
    blocks = adversarial_blocks(g, seed)
    per_tok = hkv * d // 16
    ntok = -(-blocks.shape[0] // per_tok)
    ntok = -(-ntok // 16) * 16
    nreq = ntok // 16
    cfg = W.custom_workload(seed=seed, batch=nreq, kv_lens=(16,) * nreq, qo_len=16,
                            num_qo_heads=hq, num_kv_heads=hkv, head_dim_qk=d,
                            head_dim_vo=d, causal=True)
    batch = W.make_batch(cfg)
    rng = np.random.default_rng(seed + 1)
    pad = ntok * per_tok - blocks.shape[0]
    kb = np.concatenate([blocks, bf16(rng.standard_normal((pad, 16)) * g)])
    vb = kb[rng.permutation(kb.shape[0])]
    assert batch.prefix.k.shape[0] == 0 and batch.new.k.shape[0] == ntok
    batch.new.k = torch.tensor(kb.reshape(ntok, hkv, d)).to(torch.bfloat16)
    batch.new.v = torch.tensor(vb.reshape(ntok, hkv, d)).to(torch.bfloat16)
    batch.k_global_scale = g
    batch.v_global_scale = g
    return batch


def oracle_bytes(batch):
    oc, _ = O.cache_from_batch(batch, "HND")
    return oc


@pytest.mark.parametrize("gname", list(GLOBAL_SCALES))
def test_quantize_append_adversarial(gname):
    g = GLOBAL_SCALES[gname]
    batch = adversarial_batch(g, seed=100 + list(GLOBAL_SCALES).index(gname))
    gc = H.GpuCase(batch)
    assert int(gc.flags.item()) == 0
    H.compare_cache_bytes(gc.cache, oracle_bytes(batch))


@pytest.mark.parametrize("kernel", [1, 3])
@pytest.mark.parametrize("gname", list(GLOBAL_SCALES))
def test_fused_append_adversarial(gname, kernel):
    g = GLOBAL_SCALES[gname]
    batch = adversarial_batch(g, seed=200 + list(GLOBAL_SCALES).index(gname))
    gc = H.GpuCase(batch, append=False, kernel=kernel)
    assert gc.plan.info.kernel == kernel
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) + batch.new.positions.long())
    out, lse = N.nvfp4kv_decode_append_run(gc.plan, batch.new.k[order].cuda(),
                                           batch.new.v[order].cuda(), gc.q, gc.cache,
                                           gc.kv_indices, batch.sm_scale)
    torch.cuda.synchronize()
    assert N.nvfp4kv_workspace_flags(gc.plan) == 0
    H.compare_cache_bytes(gc.cache, oracle_bytes(batch))
    # attention over such blocks is only checked for being written and finite
    # here (values reach 6 * 448 * 2^60); its accuracy is the parity tests'
    assert not torch.isnan(lse).any()
    assert bool(torch.isfinite(out.float()).all())
