"""Pins of the float64 CPU oracle against things other than itself.

Each pin uses an independent route: torch's float8 conversions (a library
routine), exact rational arithmetic (fractions.Fraction), torch SDPA in
float64, closed forms, values the pages print (tests/golden/), and
invariances.  A plausible slip in the oracle (a wrong bias, a nibble swap, a
dropped scale, a wrong tie rule, a wrong kv-head mapping, a top-left causal
mask, a log2 lse) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = (s.strip() for s in line.split("=", 1))
                vals[k] = float(int(v, 16)) if v.startswith("0x") else float(v)
            else:
                a, b = line.split()
                vals[int(a)] = float(b)
    return vals


# ---- scalar formats ------------------------------------------------------

def minifloat(bits, ebits, mbits, bias, ieee_specials):
    """Generic sign/exponent/mantissa decoder (validated below on two library
    formats, then used to pin the e2m1 table)."""
    s = (bits >> (ebits + mbits)) & 1
    e = (bits >> mbits) & ((1 << ebits) - 1)
    m = bits & ((1 << mbits) - 1)
    if ieee_specials and e == (1 << ebits) - 1:
        return (math.nan if m else math.inf) * (-1 if s else 1)
    if e == 0:
        mag = math.ldexp(m / (1 << mbits), 1 - bias)
    else:
        mag = math.ldexp(1 + m / (1 << mbits), e - bias)
    return -mag if s else mag


def test_generic_decoder_matches_torch_float8():
    b = torch.arange(256, dtype=torch.uint8)
    e5 = b.view(torch.float8_e5m2).double().tolist()
    for i in range(256):
        ref = minifloat(i, 5, 2, 15, True)
        assert (math.isnan(ref) and math.isnan(e5[i])) or ref == e5[i]
    e4 = b.view(torch.float8_e4m3fn).double().tolist()
    for i in range(256):
        if (i & 0x7F) == 0x7F:
            assert math.isnan(e4[i])
        else:
            assert minifloat(i, 4, 3, 7, False) == e4[i]


def test_e4m3_table_matches_torch():
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().tolist()
    for i in range(256):
        v = O.e4m3_value(i)
        if (i & 0x7F) == 0x7F:
            assert math.isnan(v)
        else:
            assert v == e4[i], i


def test_e2m1_table():
    grid = [O.e2m1_value(c) for c in range(16)]
    for c in range(16):
        assert grid[c] == minifloat(c, 2, 1, 1, False)
    # largest e2m1 magnitude is 6: the block recipe divides amax by 6
    assert max(grid) == 6.0 and min(grid) == -6.0
    assert sorted(set(abs(x) for x in grid)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _bf16_values():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).double()
    return v[torch.isfinite(v)].tolist()


def test_e4m3_encode_matches_torch_rne():
    # torch's float32 -> float8_e4m3fn conversion is round-to-nearest-even and
    # non-saturating (>= 464 becomes NaN); compare wherever it is finite, on
    # every finite bf16 value and on the exact midpoints and their fp32
    # neighbours.
    vals = [x for x in _bf16_values() if abs(x) < 464]
    mids = []
    fin = [O.e4m3_value(i) for i in range(0x7F)]
    for a, b in zip(fin, fin[1:]):
        m = (a + b) / 2
        mids += [m, float(np.nextafter(np.float32(m), np.float32(1e9))),
                 float(np.nextafter(np.float32(m), np.float32(0)))]
    xs = vals + mids + [-m for m in mids]
    ref = torch.tensor(xs, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [O.e4m3_encode(float(np.float32(x))) for x in xs]
    bad = [(x, r, g) for x, r, g in zip(xs, ref, got) if r != g]
    assert not bad, bad[:10]


def test_e4m3_encode_saturates():
    for x in (448.0, 463.99, 464.0, 480.0, 1e6, 1e300):
        assert O.e4m3_encode(x) == 0x7E
        assert O.e4m3_encode(-x) == 0xFE


def _nearest_even(x, grid_codes):
    """Exact nearest grid value (Fraction arithmetic), ties to the even code."""
    best = None
    for c, v in grid_codes:
        d = abs(Fraction(x) - Fraction(v))
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e2m1_encode_brute_force():
    pos = [(c, O.e2m1_value(c)) for c in range(8)]
    xs = [x for x in _bf16_values() if abs(x) <= 16]
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        xs += [m, math.nextafter(m, 0), math.nextafter(m, 9)]
    for x in xs:
        want = _nearest_even(min(abs(x), 6.0), pos) | (8 if math.copysign(1, x) < 0 else 0)
        assert O.e2m1_encode(x) == want, x


def test_e2m1_ties_table():
    # round-half-to-even on the code: 0.25->0, 0.75->1, 1.25->1, 1.75->2,
    # 2.5->2, 3.5->4, 5->4; >6 saturates; the sign of x is kept (-0.1 -> -0)
    for x, v in [(0.25, 0), (0.75, 1), (1.25, 1), (1.75, 2), (2.5, 2), (3.5, 4),
                 (5.0, 4), (7.0, 6), (100.0, 6)]:
        assert O.e2m1_value(O.e2m1_encode(x)) == v
        assert O.e2m1_value(O.e2m1_encode(-x)) == -v
    assert O.e2m1_encode(-0.1) == 8 and O.e2m1_encode(0.1) == 0
    assert O.e2m1_encode(-0.0) == 8


# ---- block quantiser -----------------------------------------------------

def exact_block(x, g):
    """Exact-real reference of the block recipe with Fractions."""
    e4 = [(i, O.e4m3_value(i)) for i in range(0x7F)]
    e2 = [(c, O.e2m1_value(c)) for c in range(8)]
    g = Fraction(g)
    amax = max(abs(Fraction(v)) for v in x)
    t = amax / (6 * g)
    sf = 0x7E if t > 448 else _nearest_even(t, e4)
    s = Fraction(O.e4m3_value(sf))
    codes = []
    for v in x:
        sign = 8 if math.copysign(1, v) < 0 else 0
        if s == 0:
            codes.append(sign)
            continue
        q = abs(Fraction(v)) / (s * g)
        codes.append((7 if q > 6 else _nearest_even(q, e2)) | sign)
    return [codes[2 * k] | (codes[2 * k + 1] << 4) for k in range(8)], sf


@pytest.mark.parametrize("g", [1.0, 0.0187872014939785, 1.0 / 2688, 3.7e-3, 250.0])
def test_block_quantiser_exact_rational(g):
    g = float(np.float32(g))
    rng = np.random.default_rng(7)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-4, 3)
        x = torch.tensor(rng.standard_normal(16) * scale, dtype=torch.float32)
        x = x.to(torch.bfloat16).double().numpy()
        if trial % 7 == 0:  # adversarial: exact ties x = midpoint * s * g
            s = O.e4m3_value(O.e4m3_encode(np.abs(x).max() / (6 * g)))
            if s > 0:
                mids = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], 16)
                x = torch.tensor(mids * s * g * rng.choice([-1, 1], 16)).to(torch.bfloat16).double().numpy()
        packed, sf = O.quantize_block16(x, g)
        want_p, want_sf = exact_block(x.tolist(), g)
        assert sf == want_sf
        assert packed.tolist() == want_p


def test_block_roundtrip_and_nibble_order():
    # x built from known codes with one |code| = 6 and a scale s: amax/6 = s,
    # so quantisation must return exactly those codes, low nibble = even index
    rng = np.random.default_rng(3)
    for _ in range(200):
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = rng.choice([7, 15])
        sfb = int(rng.integers(1, 0x7F))
        s = O.e4m3_value(sfb)
        x = np.array([O.e2m1_value(int(c)) * s for c in codes])
        packed, sf = O.quantize_block16(x, 1.0)
        assert sf == sfb
        exp = [int(codes[2 * k] | (codes[2 * k + 1] << 4)) for k in range(8)]
        # zero codes keep the sign of x; +0 and -0 are both value 0
        got = packed.tolist()
        for k in range(8):
            for half in (0, 1):
                gc = (got[k] >> (4 * half)) & 15
                ec = (exp[k] >> (4 * half)) & 15
                assert O.e2m1_value(gc) == O.e2m1_value(ec)
                if ec & 7:
                    assert gc == ec


def test_block_zero_and_negative_zero():
    packed, sf = O.quantize_block16(np.zeros(16), 1.0)
    assert sf == 0 and packed.tolist() == [0] * 8
    packed, sf = O.quantize_block16(-np.zeros(16), 1.0)
    assert sf == 0 and packed.tolist() == [0x88] * 8
    # underflowing scale: amax/(6g) below half the smallest subnormal
    packed, sf = O.quantize_block16(np.full(16, 1e-5), 1.0)
    assert sf == 0 and packed.tolist() == [0] * 8


def test_worked_example_v_ones():
    gold = read_golden("v_ones_probe.txt")
    packed, sf = O.quantize_block16(np.ones(16), gold["global_scale"])
    assert sf == gold["scale_byte"]
    assert O.e4m3_value(sf) == gold["scale"]
    assert packed.tolist() == [int(gold["code"]) * 17] * 8
    deq = O.e2m1_value(int(gold["code"])) * O.e4m3_value(sf) * gold["global_scale"]
    assert deq == gold["dequant"]
    assert round(deq, 3) == gold["printed_fixed"]
    assert round(deq / 2, 4) == gold["printed_half"]


def test_second_closed_form_scale_448():
    g = float(np.float32(1.0 / (6 * 448)))
    packed, sf = O.quantize_block16(np.ones(16), g)
    assert O.e4m3_value(sf) == 448.0 and packed.tolist() == [0x77] * 8
    assert 6 * 448.0 * g == pytest.approx(1.0, rel=1e-7)


# ---- attention -----------------------------------------------------------

def small_batch(kv_lens=(37, 100), qo_len=1, Hq=4, Hkv=1, Dk=128, Dv=128,
                causal=False, seed=11, extra_pages=0, **kw):
    cfg = W.custom_workload(seed=seed, batch=len(kv_lens), qo_len=qo_len,
                            num_qo_heads=Hq, num_kv_heads=Hkv, head_dim_qk=Dk,
                            head_dim_vo=Dv, kv_lens=kv_lens, causal=causal, **kw)
    return W.make_batch(cfg, extra_pages=extra_pages)


def dense_kv(cache, pt, b, h, L):
    """Dequantised K/V rows of request b, kv head h, in token order."""
    P = cache.layout.page_size
    K, V = [], []
    for j in range(L):
        page = int(pt.kv_indices[pt.kv_indptr[b] + j // P])
        K.append(O.dequant_row(cache, 0, page, j % P, h))
        V.append(O.dequant_row(cache, 1, page, j % P, h))
    return torch.tensor(np.array(K)), torch.tensor(np.array(V))


@pytest.mark.parametrize("causal,qo_len,Hq,Hkv,Dk,Dv,layout", [
    (False, 1, 4, 1, 128, 128, "HND"),
    (False, 1, 8, 2, 64, 64, "NHD"),
    (True, 5, 6, 2, 64, 32, "HND"),
    (True, 3, 8, 1, 128, 256, "NHD"),
])
def test_attention_matches_sdpa_float64(causal, qo_len, Hq, Hkv, Dk, Dv, layout):
    batch = small_batch((37, 100, 16), qo_len, Hq, Hkv, Dk, Dv, causal)
    cache, pt = O.cache_from_batch(batch, layout)
    out, lse = O.attention(cache, pt, batch.qo_indptr, batch.q, Hq, causal,
                           batch.sm_scale)
    G = Hq // Hkv
    for b, L in enumerate(batch.kv_lens):
        q0 = b * qo_len
        q = batch.q[q0:q0 + qo_len].double()                 # [n, Hq, Dk]
        for h in range(Hkv):
            K, V = dense_kv(cache, pt, b, h, L)
            qh = q[:, h * G:(h + 1) * G].transpose(0, 1)     # [G, n, Dk]
            i = torch.arange(qo_len)[:, None]
            j = torch.arange(L)[None, :]
            mask = (j <= L - qo_len + i) if causal else torch.ones(qo_len, L, dtype=torch.bool)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qh, K[None], V[None], attn_mask=mask, scale=batch.sm_scale)
            s = (qh @ K.T) * batch.sm_scale
            ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
            got = torch.tensor(out[q0:q0 + qo_len, h * G:(h + 1) * G]).transpose(0, 1)
            got_lse = torch.tensor(lse[q0:q0 + qo_len, h * G:(h + 1) * G]).T
            assert torch.allclose(got, ref, atol=1e-12, rtol=0)
            assert torch.allclose(got_lse, ref_lse, atol=1e-12, rtol=0)


def test_dense_rows_match_block_quantiser():
    # the paged store/lookup of a token reproduces the block recipe applied to
    # that token's bf16 row
    batch = small_batch((37, 100), Dk=64, Dv=32)
    cache, pt = O.cache_from_batch(batch, "NHD")
    P = 16
    for t in range(0, batch.prefix.k.shape[0], 7):
        b = int(batch.prefix.batch_idx[t]); pos = int(batch.prefix.positions[t])
        page = int(pt.kv_indices[pt.kv_indptr[b] + pos // P])
        row = O.dequant_row(cache, 0, page, pos % P, 0)
        x = batch.prefix.k[t, 0].double().numpy()
        for j in range(4):
            packed, sf = O.quantize_block16(x[16 * j:16 * j + 16], 1.0)
            vals = []
            for byte in packed:
                vals += [O.e2m1_value(int(byte) & 15), O.e2m1_value(int(byte) >> 4)]
            assert np.array_equal(row[16 * j:16 * j + 16], np.array(vals) * O.e4m3_value(sf))


def test_uniform_score_probe_q_zero():
    gold = read_golden("uniform_lse.txt")
    batch = small_batch((37, 100, 16, 1), qo_len=1)
    batch.q.zero_()
    cache, pt = O.cache_from_batch(batch)
    out, lse = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, False, batch.sm_scale)
    for b, L in enumerate(batch.kv_lens):
        _, V = dense_kv(cache, pt, b, 0, L)
        mean = V.sum(0) / L
        assert np.allclose(out[b], mean.numpy()[None], atol=1e-15, rtol=0)
        assert np.all(lse[b] == gold[L])
        assert gold[L] == pytest.approx(math.log(L), abs=1e-15)


def test_v_ones_probe_through_attention():
    gold = read_golden("v_ones_probe.txt")
    batch = small_batch((37, 100), qo_len=3, causal=True)
    for ts in (batch.prefix, batch.new):
        ts.v.fill_(1.0)
    cache, pt = O.cache_from_batch(batch)
    out, _ = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, True, batch.sm_scale)
    assert np.allclose(out, gold["dequant"], atol=1e-14, rtol=0)


def test_distinct_k_and_v_global_scales():
    # V must be dequantised with its own global scale (the pages' decode test
    # once used K's): V = ones with g_V = 1/(6*448) dequantises to exactly 1,
    # while K keeps g_K = 1 (scores unchanged), so the output is exactly 1.
    batch = small_batch((37, 100), qo_len=2, causal=True)
    for ts in (batch.prefix, batch.new):
        ts.v.fill_(1.0)
    batch.k_global_scale = 1.0
    batch.v_global_scale = float(np.float32(1.0 / (6 * 448)))
    cache, pt = O.cache_from_batch(batch)
    out, _ = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, True, batch.sm_scale)
    assert np.allclose(out, 1.0, atol=1e-6, rtol=0)
    # and the K scale enters the scores: scaling g_K by 2 (codes unchanged)
    # equals doubling sm_scale
    batch2 = small_batch((37, 100), qo_len=2, causal=True)
    c1, pt1 = O.cache_from_batch(batch2)
    o_ref, l_ref = O.attention(c1, pt1, batch2.qo_indptr, batch2.q, 4, True,
                               2 * batch2.sm_scale)
    c1.k_global_scale = 2.0
    c1._s.k_global_scale = 2.0
    o2, l2 = O.attention(c1, pt1, batch2.qo_indptr, batch2.q, 4, True, batch2.sm_scale)
    assert np.allclose(o2, o_ref, atol=1e-13) and np.allclose(l2, l_ref, atol=1e-13)


def test_single_key_closed_form():
    batch = small_batch((1, 17), qo_len=1)
    cache, pt = O.cache_from_batch(batch)
    out, lse = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, False, batch.sm_scale)
    K, V = dense_kv(cache, pt, 0, 0, 1)
    s = batch.q[0].double() @ K[0] * batch.sm_scale
    assert np.allclose(out[0], V[0].numpy()[None], atol=0, rtol=0)
    assert np.allclose(lse[0], s.numpy(), atol=1e-13, rtol=0)


@pytest.mark.parametrize("causal,qo_len", [(False, 1), (True, 7)])
def test_split_invariance(causal, qo_len):
    batch = small_batch((37, 100, 250), qo_len=qo_len, Hq=4, Hkv=2, causal=causal)
    cache, pt = O.cache_from_batch(batch)
    ref, ref_lse = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, causal, batch.sm_scale)
    for chunk in (16, 32, 48, 112, 250):
        out, lse = O.attention(cache, pt, batch.qo_indptr, batch.q, 4, causal,
                               batch.sm_scale, chunk_tokens=chunk)
        assert np.allclose(out, ref, atol=1e-12, rtol=0)
        assert np.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_page_order_invariance_and_poison():
    batch = small_batch((37, 100, 61), qo_len=2, causal=True, extra_pages=5)
    c1, pt1 = O.cache_from_batch(batch, fill=0xFF)   # unused pages: NaN scales
    o1, l1 = O.attention(c1, pt1, batch.qo_indptr, batch.q, 4, True, batch.sm_scale)
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    # permute the physical pages (a fresh page table over the same tokens)
    perm = torch.randperm(batch.num_pages, generator=torch.Generator().manual_seed(9))
    batch.kv_indices = perm[batch.kv_indices.long()].to(torch.int32)
    c2, pt2 = O.cache_from_batch(batch, fill=0xFF)
    o2, l2 = O.attention(c2, pt2, batch.qo_indptr, batch.q, 4, True, batch.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gqa_head_mapping():
    # query head h must attend kv head h // G: give kv head 1 V = ones and kv
    # head 0 V = zeros; heads 0..G-1 see 0, heads G..2G-1 see the ones value
    batch = small_batch((37, 50), qo_len=1, Hq=6, Hkv=2)
    for ts in (batch.prefix, batch.new):
        ts.v[:, 0] = 0.0
        ts.v[:, 1] = 1.0
    cache, pt = O.cache_from_batch(batch)
    out, _ = O.attention(cache, pt, batch.qo_indptr, batch.q, 6, False, batch.sm_scale)
    assert np.all(out[:, :3] == 0.0)
    assert np.allclose(out[:, 3:], 1.03125, atol=1e-14)


def test_merge_states_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((3, 8))
    out, lse = O.merge_states(o[:1], [0.7])
    assert np.array_equal(out, o[0]) and lse == 0.7
    out, lse = O.merge_states(o[:2], [1.5, 1.5])
    assert np.allclose(out, (o[0] + o[1]) / 2, atol=1e-15)
    assert lse == pytest.approx(1.5 + math.log(2), abs=1e-15)
    out, lse = O.merge_states(o, [-math.inf] * 3)
    assert np.all(out == 0) and lse == -math.inf
    out, lse = O.merge_states(o, [-math.inf, 2.0, -math.inf])
    assert np.allclose(out, o[1], atol=0) and lse == 2.0
    # weights are softmax of lse
    ls = np.array([0.3, -1.2, 2.5])
    w = np.exp(ls - ls.max()); w /= w.sum()
    out, lse = O.merge_states(o, ls)
    assert np.allclose(out, w @ o, atol=1e-14)
    assert lse == pytest.approx(np.log(np.exp(ls).sum()), abs=1e-14)


def test_append_rejects_out_of_range():
    batch = small_batch((37, 100))
    cache = O.Cache(batch.cache_layout(), 1.0, 1.0)
    pt = O.PageTable.of(batch)
    bad = W.TokenSet(torch.tensor([0], dtype=torch.int32),
                     torch.tensor([37], dtype=torch.int32),
                     batch.new.k[:1], batch.new.v[:1])
    assert O.quantize_append(cache, pt, bad) == 2
    assert not cache.bufs["k_data"].any()


@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_page_size_one_matches_sixteen(layout):
    """The oracle reaches every token through the page table at any page size
    (page "Re-enable split-KV for NVFP4 KV cache in prefill path": the paged
    layout with an indptr of pages and a last-page length): the same tokens
    stored one per page, in permuted pages, give bit-identical float64
    attention and the same stored bytes per token as 16-token pages."""
    cfg = W.custom_workload(seed=11, batch=3, qo_len=2, num_qo_heads=8, num_kv_heads=2,
                            kv_lens=(37, 100, 16), causal=True)
    batch = W.make_batch(cfg)
    c16, pt16 = O.cache_from_batch(batch, layout)
    out16, lse16 = O.attention(c16, pt16, batch.qo_indptr, batch.q, cfg.num_qo_heads,
                               True, batch.sm_scale)

    lens = [int(x) for x in batch.kv_lens]
    total = sum(lens)
    perm = np.random.default_rng(5).permutation(total).astype(np.int32)
    pt1 = O.PageTable(perm, np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                      np.ones(len(lens), np.int32))
    lay1 = W.CacheLayout(layout, total, 1, cfg.num_kv_heads, cfg.head_dim_qk,
                         cfg.head_dim_vo)
    c1 = O.Cache(lay1, batch.k_global_scale, batch.v_global_scale, fill=0xFF)
    assert O.quantize_append(c1, pt1, batch.prefix) == 0
    assert O.quantize_append(c1, pt1, batch.new) == 0
    out1, lse1 = O.attention(c1, pt1, batch.qo_indptr, batch.q, cfg.num_qo_heads, True,
                             batch.sm_scale)
    assert np.array_equal(out1, out16) and np.array_equal(lse1, lse16)

    # token (b, pos) of kv head h: page perm[indptr_b + pos] slot 0 against
    # page kv_indices[indptr16_b + pos // 16] slot pos % 16
    kvi, kvp = batch.kv_indices.numpy(), batch.kv_indptr.numpy()
    off = np.concatenate([[0], np.cumsum(lens)])
    for b, pos, h in [(0, 0, 0), (0, 36, 1), (1, 17, 0), (1, 99, 1), (2, 15, 0)]:
        for which in (0, 1):
            a = O.dequant_row(c1, which, int(perm[off[b] + pos]), 0, h)
            r = O.dequant_row(c16, which, int(kvi[kvp[b] + pos // 16]), pos % 16, h)
            assert np.array_equal(a, r)


# ---- attention with FP4 query and probabilities ---------------------------
# Page "fix(attention): correct SM120 NVFP4 qk_correction layout, row-sum
# reduction, and lse", description: Q, K, V and P quantised to FP4; the row
# sum carries the FP4 P quantisation factor, which lse drops; the uniform-score
# V = ones probe returns the V-quantisation value; uniform scores give
# lse = ln(seq_len).

P_SCALE = 448.0 * 6.0   # E4M3 maximum x e2m1 maximum


def fp4_block_values(x):
    """Exact-real NVFP4 (global scale 1) of 16 values, as values."""
    packed, sf = exact_block([float(v) for v in x], 1.0)
    s = O.e4m3_value(sf)
    vals = []
    for byte in packed:
        vals += [O.e2m1_value(byte & 15) * s, O.e2m1_value(byte >> 4) * s]
    return vals


def test_fp4qp_uniform_score_v_ones_probe():
    gold_v = read_golden("v_ones_probe.txt")
    gold_l = read_golden("uniform_lse.txt")
    batch = small_batch((37, 100, 16, 1), qo_len=1)
    batch.q.zero_()
    for ts in (batch.prefix, batch.new):
        ts.v.fill_(1.0)
    cache, pt = O.cache_from_batch(batch)
    out, lse = O.attention_fp4qp(cache, pt, batch.qo_indptr, batch.q, 4, False,
                                 batch.sm_scale)
    assert np.all(out == gold_v["dequant"])
    for b, L in enumerate(batch.kv_lens):
        assert np.all(lse[b] == gold_l[L])


def test_fp4qp_reduces_to_exact_attention_when_q_and_p_are_fp4_values():
    # q = 1.03125 e_0 is its own NVFP4 value (scale E4M3(1.03125/6) = 0.171875,
    # code 6); K rows k_j = c_j e_0 with c_j in {1.5, 0.75, 0} are their own
    # NVFP4 values; sm_scale = ln 2 / (1.03125 * 0.75) makes the scores
    # {2 ln 2, ln 2, 0}, so p in {1, 1/2, 1/4} and 2688 p in {2688, 1344, 672}
    # = 448 x {6, 3, 1.5}: every quantisation is exact and the method is plain
    # attention.
    batch = small_batch((37, 21), qo_len=1, Hq=2, Hkv=1, Dk=32, Dv=32)
    batch.q.zero_()
    batch.q[:, :, 0] = 1.03125
    rng = np.random.default_rng(5)
    for ts in (batch.prefix, batch.new):
        ts.k.zero_()
        ts.k[:, :, 0] = torch.tensor(rng.choice([1.5, 0.75, 0.0], ts.k.shape[0]),
                                     dtype=torch.bfloat16)[:, None]
    sm = math.log(2.0) / (1.03125 * 0.75)
    cache, pt = O.cache_from_batch(batch)
    ref, ref_lse = O.attention(cache, pt, batch.qo_indptr, batch.q, 2, False, sm)
    out, lse = O.attention_fp4qp(cache, pt, batch.qo_indptr, batch.q, 2, False, sm)
    assert np.allclose(out, ref, atol=1e-14, rtol=0)
    assert np.allclose(lse, ref_lse, atol=1e-14, rtol=0)


def test_fp4qp_lse_is_that_of_the_quantised_query():
    # lse does not depend on P's quantisation: it is the plain log-sum-exp of
    # the scores of the quantised query.  The quantised query is exact in bf16
    # (2 + 3 significant bits), so the exact attention of that query gives it,
    # and quantising the query again changes nothing.
    batch = small_batch((37, 100, 5), qo_len=2, Hq=4, Hkv=2, Dk=64, Dv=32, causal=True)
    cache, pt = O.cache_from_batch(batch)
    qh = batch.q.clone()
    flat = qh.double().reshape(-1, 16).numpy()
    qh = torch.tensor(np.array([fp4_block_values(r) for r in flat])).reshape(qh.shape)
    assert torch.equal(qh.to(torch.bfloat16).double(), qh)
    qh = qh.to(torch.bfloat16)
    out1, lse1 = O.attention_fp4qp(cache, pt, batch.qo_indptr, batch.q, 4, True, batch.sm_scale)
    out2, lse2 = O.attention_fp4qp(cache, pt, batch.qo_indptr, qh, 4, True, batch.sm_scale)
    _, ref_lse = O.attention(cache, pt, batch.qo_indptr, qh, 4, True, batch.sm_scale)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    assert np.allclose(lse1, ref_lse, atol=1e-13, rtol=0)


@pytest.mark.parametrize("causal,qo_len", [(False, 1), (True, 3)])
def test_fp4qp_brute_force_small(causal, qo_len):
    # every quantisation by the exact rational search over E4M3 and e2m1
    # values; scores, maxima and sums accumulated in the oracle's order
    Hq, Hkv, Dk, Dv = 2, 1, 32, 16
    batch = small_batch((37, 20), qo_len=qo_len, Hq=Hq, Hkv=Hkv, Dk=Dk, Dv=Dv,
                        causal=causal, seed=23)
    cache, pt = O.cache_from_batch(batch)
    out, lse = O.attention_fp4qp(cache, pt, batch.qo_indptr, batch.q, Hq, causal,
                                 batch.sm_scale)
    for b, L in enumerate(batch.kv_lens):
        K, V = dense_kv(cache, pt, b, 0, L)
        K, V = K.numpy(), V.numpy()
        for i in range(qo_len):
            row = b * qo_len + i
            lim = L - qo_len + i if causal else L - 1
            for h in range(Hq):
                x = batch.q[row, h].double().numpy()
                qv = sum((fp4_block_values(x[k:k + 16]) for k in range(0, Dk, 16)), [])
                s = []
                for j in range(L):
                    acc = 0.0
                    for d in range(Dk):
                        acc += qv[d] * K[j, d]
                    s.append(batch.sm_scale * acc)
                m = max(s[:lim + 1])
                z = 0.0
                for j in range(lim + 1):
                    z += math.exp(s[j] - m)
                o = np.zeros(Dv)
                for blk in range(0, L, 16):
                    pp = [P_SCALE * math.exp(s[j] - m) if j < L and j <= lim else 0.0
                          for j in range(blk, blk + 16)]
                    ph = fp4_block_values(pp)
                    for t in range(16):
                        if blk + t < L:
                            o += ph[t] * V[blk + t]
                assert np.allclose(out[row, h], o / (P_SCALE * z), atol=1e-13, rtol=0)
                assert lse[row, h] == pytest.approx(m + math.log(z), abs=1e-13)
