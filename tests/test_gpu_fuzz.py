"""Randomised parity sweeps through the C ABI against the float64 oracle:
seeded draws of batch, heads and GQA ratio, lengths (ragged, empty),
head_dim, causality, the variants (sliding window, soft-capping, ALiBi),
packed sequences, paged or contiguous caches, block sizes, split counts and
decode with append.
Each case is small enough for the oracle's full result, and every element is
compared."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
import oracle
from gpu_util import compare, nan_like

pytestmark = pytest.mark.gpu


def _variant(rng, n_max):
    """One of: none, a window, a soft cap, ALiBi (with or without a window)."""
    kind = int(rng.integers(0, 5))
    if kind == 1:
        return {"window_left": int(rng.integers(0, max(1, n_max)))}
    if kind == 2:
        return {"softcap": float(rng.uniform(1.0, 50.0))}
    if kind == 3:
        return {"alibi": True}
    if kind == 4:
        return {"alibi": True, "window_left": int(rng.integers(0, max(1, n_max)))}
    return {}


def _split(variant, hq, dev):
    """(kwargs for the library, kwargs for the oracle)."""
    kw = {k: v for k, v in variant.items() if k != "alibi"}
    okw = dict(kw)
    if variant.get("alibi"):
        sl = torch.tensor([2.0 ** (-(h % 8 + 1)) for h in range(hq)], dtype=torch.float32)
        kw["alibi_slopes"] = sl.to(dev)
        okw["alibi_slopes"] = sl.tolist()
    return kw, okw


@pytest.mark.parametrize("case", range(48))
def test_prefill_fuzz(dev, case):
    rng = np.random.default_rng(1000 + case)
    d = int(rng.choice([64, 128, 256]))
    B = int(rng.integers(1, 4))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 3, 4, 7, 8]))
    N = int(rng.integers(1, 1201))
    causal = bool(rng.integers(0, 2))
    variant = _variant(rng, N)
    x = W.make_prefill(B, hq, hkv, N, d, seed=case, spike_frac=0.01 * int(rng.integers(0, 2)),
                       causal=causal)
    kw, okw = _split(variant, hq, dev)
    o, lse = nan_like((B, hq, N, d), dev), nan_like((B, hq, N), dev)
    attn.prefill(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.scale, causal, out=o, lse=lse, **kw)
    attn.check_device_status()
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal, **okw)
    what = f"case {case}: B{B} H{hq}/{hkv} N{N} d{d} causal={causal} {variant}"
    compare(o, lse, o_ref, lse_ref, what)
    # the same call with a bf16 O: the fp32 O rounded once, bit for bit
    o16, l16 = attn.prefill(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.scale, causal,
                            out_dtype=torch.bfloat16, **kw)
    attn.check_device_status()
    assert torch.equal(o16, o.to(torch.bfloat16)) and torch.equal(l16, lse), what + " (bf16 O)"


@pytest.mark.parametrize("case", range(32))
def test_prefill_varlen_fuzz(dev, case):
    rng = np.random.default_rng(2000 + case)
    d = int(rng.choice([64, 128, 256]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4, 7]))
    n_seqs = int(rng.integers(1, 9))
    lens = [int(n) for n in rng.integers(0, 601, n_seqs)]
    causal = bool(rng.integers(0, 2))
    variant = _variant(rng, max(lens) if lens else 1)
    x = W.make_prefill_varlen(lens, hq, hkv, d, seed=case, extra_rows=int(rng.integers(0, 5)),
                              causal=causal)
    kw, okw = _split(variant, hq, dev)
    n_q, T, _ = x.q.shape
    o, lse = nan_like((n_q, T, d), dev), nan_like((n_q, T), dev)
    attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev), x.scale,
                        causal, out=o, lse=lse, **kw)
    attn.check_device_status()
    o_ref, lse_ref = oracle.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, x.scale, causal, **okw)
    T0 = int(x.cu_seqlens[-1])
    what = f"case {case}: lens {lens} H{hq}/{hkv} d{d} causal={causal} {variant}"
    compare(o[:, :T0], lse[:, :T0], o_ref[:, :T0], lse_ref[:, :T0], what)
    assert torch.isnan(o[:, T0:]).all() and torch.isnan(lse[:, T0:]).all()
    o16 = torch.full((n_q, T, d), float("nan"), dtype=torch.bfloat16, device=dev)
    attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev), x.scale,
                        causal, out=o16, out_dtype=torch.bfloat16, **kw)
    attn.check_device_status()
    assert torch.equal(o16[:, :T0], o[:, :T0].to(torch.bfloat16)), what + " (bf16 O)"
    assert torch.isnan(o16[:, T0:].float()).all(), what + " (bf16 O past the end)"


@pytest.mark.parametrize("case", range(48))
def test_decode_fuzz(dev, case):
    rng = np.random.default_rng(3000 + case)
    d = int(rng.choice([64, 128, 256]))
    B = int(rng.integers(1, 5))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4, 7, 8, 16, 24]))
    lens = [int(n) for n in rng.integers(0, 3001, B)]
    paged = bool(rng.integers(0, 2))
    variant = _variant(rng, max(lens) + 1)
    if paged:
        bs = int(rng.choice([16, 32, 64, 8, 24]))
        dd = W.make_decode_paged(B, hq, hkv, d, lens, block_size=bs, seed=case,
                                 extra_blocks=int(rng.integers(0, 3)))
    else:
        L = max(lens) + int(rng.integers(0, 40))
        dd = W.make_decode_contiguous(B, hq, hkv, d, max(L, 1), seed=case, max_kv_len=max(L, 1))
        dd.kv_lens = torch.tensor(lens, dtype=torch.int32)
    S = int(rng.choice([1, 3, 16, 64])) if rng.integers(0, 2) else attn.decode_num_splits(
        B, hkv, max(max(lens), 1))
    kw, okw = _split(variant, hq, dev)
    bt = dd.block_table.to(dev) if dd.block_table is not None else None
    op, lp = nan_like((S, B, hq, d), dev), nan_like((S, B, hq), dev)
    attn.decode_splitkv(dd.q.to(dev), dd.k_cache.to(dev), dd.v_cache.to(dev), dd.kv_lens.to(dev),
                        bt, num_splits=S, max_kv_len=dd.max_kv_len, scale=dd.scale,
                        o_partial=op, lse_partial=lp, **kw)
    o, lse = nan_like((B, hq, d), dev), nan_like((B, hq), dev)
    attn.combine(op, lp, out=o, lse=lse)
    attn.check_device_status()
    o_ref, lse_ref = oracle.decode(dd.q, dd.k_cache, dd.v_cache, dd.block_table, lens, dd.scale,
                                   dd.block_size, **okw)
    compare(o, lse, o_ref, lse_ref,
            f"case {case}: B{B} H{hq}/{hkv} d{d} lens {lens} paged={paged} S={S} {variant}")


@pytest.mark.parametrize("case", range(24))
def test_decode_append_fuzz(dev, case):
    """Decode that first writes each sequence's new key and value at position
    kv_lens[b]: the combined result against the oracle's decode_append, and
    the caches afterwards bit for bit."""
    rng = np.random.default_rng(4000 + case)
    d = int(rng.choice([64, 128, 256]))
    B = int(rng.integers(1, 5))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4, 7, 8]))
    lens = [int(n) for n in rng.integers(0, 2001, B)]
    paged = bool(rng.integers(0, 2))
    variant = _variant(rng, max(lens) + 2)
    if paged:
        bs = int(rng.choice([16, 32, 64, 8, 24]))
        dd = W.make_decode_paged(B, hq, hkv, d, [n + 1 for n in lens], block_size=bs, seed=case)
    else:
        L = max(lens) + 1 + int(rng.integers(0, 40))
        dd = W.make_decode_contiguous(B, hq, hkv, d, L, seed=case, max_kv_len=L)
    dd.kv_lens = torch.tensor(lens, dtype=torch.int32)
    g = torch.Generator().manual_seed(case)
    kn = torch.randn(B, hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, hkv, d, generator=g).to(torch.bfloat16)
    S = int(rng.choice([1, 5, 16])) if rng.integers(0, 2) else attn.decode_num_splits(
        B, hkv, max(lens) + 1)
    kw, okw = _split(variant, hq, dev)
    kc, vc = dd.k_cache.to(dev), dd.v_cache.to(dev)
    bt = dd.block_table.to(dev) if dd.block_table is not None else None
    op, lp = nan_like((S, B, hq, d), dev), nan_like((S, B, hq), dev)
    attn.decode_append_splitkv(dd.q.to(dev), kn.to(dev), vn.to(dev), kc, vc, dd.kv_lens.to(dev),
                               bt, num_splits=S, max_kv_len=dd.max_kv_len or None,
                               scale=dd.scale, o_partial=op, lse_partial=lp, **kw)
    o, lse = nan_like((B, hq, d), dev), nan_like((B, hq), dev)
    attn.combine(op, lp, out=o, lse=lse)
    attn.check_device_status()
    o_ref, lse_ref, kc_ref, vc_ref = oracle.decode_append(dd.q, kn, vn, dd.k_cache, dd.v_cache,
                                                          dd.block_table, lens, dd.scale,
                                                          dd.block_size, **okw)
    what = f"case {case}: B{B} H{hq}/{hkv} d{d} lens {lens} paged={paged} S={S} {variant}"
    compare(o, lse, o_ref, lse_ref, what)
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16)
    assert torch.equal(bits(kc), bits(kc_ref)), what + ": K cache"
    assert torch.equal(bits(vc), bits(vc_ref)), what + ": V cache"


@pytest.mark.parametrize("case", range(12))
def test_prefill_fp8_fuzz(dev, case):
    """FP8 prefill (block scales, rotation) on random shapes: LSE within 1e-3
    of exact attention on the dequantised inputs, O within the P-rounding
    bound (as the FP8 parity tests)."""
    from test_gpu_fp8 import fp8_inputs, p_rounding_sigma, signs_for
    from oracle import fp8_ref as F

    rng = np.random.default_rng(5000 + case)
    d = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 3))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4, 7]))
    N = 16 * int(rng.integers(1, 65))
    causal = bool(rng.integers(0, 2))
    x = W.make_prefill(B, hq, hkv, N, d, seed=case, causal=causal)
    signs = signs_for(d, case)
    q8, k8, v8t, qs, ks, vs = fp8_inputs(x, dev, signs)
    o, lse = attn.prefill_fp8(q8, k8, v8t, qs, ks, vs, x.scale, causal)
    attn.check_device_status()
    qz = F.quantize_for_attention(x.q, x.k, x.v, signs)
    o_ref, lse_ref = F.prefill_fp8(qz, x.scale, causal)
    what = f"case {case}: B{B} H{hq}/{hkv} N{N} d{d} causal={causal}"
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3, what
    z = np.abs(o.double().cpu().numpy() - o_ref) / (p_rounding_sigma(qz, x.scale, causal) + 1e-6)
    assert z.max() <= 6.0 and z.mean() <= 1.0, (what, z.max(), z.mean())


@pytest.mark.parametrize("case", range(8))
def test_prefill_fp8_varlen_fuzz(dev, case):
    """Packed FP8 prefill on random sequence lists (every sequence starting
    at a multiple of 16 rows; the last one of any length)."""
    import math

    from test_gpu_fp8 import packed_sigma, signs_for
    from oracle import fp8_ref as F

    rng = np.random.default_rng(6000 + case)
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    n_seqs = int(rng.integers(1, 7))
    lens = [16 * int(n) for n in rng.integers(0, 41, n_seqs - 1)] + [int(rng.integers(1, 500))]
    causal = bool(rng.integers(0, 2))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = -(-int(cu[-1]) // 16) * 16 + 16
    g = torch.Generator().manual_seed(case)
    q = torch.randn(hq, T, d, generator=g).to(torch.bfloat16)
    k = torch.randn(hkv, T, d, generator=g).to(torch.bfloat16)
    v = torch.randn(hkv, T, d, generator=g).to(torch.bfloat16)
    signs = signs_for(d, case)
    sg, cud = torch.from_numpy(signs).to(dev), torch.from_numpy(cu).to(dev)
    q8, qs = attn.quantize_fp8_varlen(q.to(dev), cud, sg)
    k8, ks = attn.quantize_fp8_varlen(k.to(dev), cud, sg)
    v8t, vs = attn.quantize_fp8(v.to(dev), None, block_rows=0, transpose=True)
    scale = 1.0 / math.sqrt(d)
    o, lse = nan_like((hq, T, d), dev), nan_like((hq, T), dev)
    attn.prefill_fp8_varlen(q8, k8, v8t, qs, ks, vs, cud, scale, causal, out=o, lse=lse)
    attn.check_device_status()
    qz = F.quantize_for_attention_varlen(q, k, v, cu, signs)
    o_ref, lse_ref = F.prefill_fp8_varlen(qz, scale, causal)
    T0 = int(cu[-1])
    what = f"case {case}: lens {lens} H{hq}/{hkv} d{d} causal={causal}"
    assert np.abs(lse[:, :T0].double().cpu().numpy() - lse_ref[:, :T0]).max() <= 1e-3, what
    z = np.abs(o[:, :T0].double().cpu().numpy() - o_ref[:, :T0]) / (
        packed_sigma(qz, scale, causal)[:, :T0] + 1e-6)
    assert z.max() <= 6.0 and z.mean() <= 1.0, (what, z.max(), z.mean())
    assert torch.isnan(o[:, T0:]).all()
