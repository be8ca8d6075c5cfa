"""Parity of the attention variants (sliding window, logit soft-capping)
through the C ABI (attn_prefill_ex, attn_decode_splitkv_ex) against the
float64 oracle: whole outputs at small sizes, sampled rows at the Qwen
shape, and decode partials under the windowed split rule."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
import oracle
from gpu_util import compare, nan_like, split_ranges

pytestmark = pytest.mark.gpu


def run_prefill(x, dev, **kw):
    B, Hq, N, D = x.q.shape
    o, lse = nan_like((B, Hq, N, D), dev), nan_like((B, Hq, N), dev)
    attn.prefill(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.scale, x.causal, out=o, lse=lse, **kw)
    attn.check_device_status()
    return o, lse


@pytest.mark.parametrize("N,Hq,Hkv,D,causal,Wl,cap", [
    (1000, 8, 2, 128, True, 0, 0.0),        # each row sees only itself
    (1000, 8, 2, 128, True, 100, 0.0),
    (777, 4, 4, 64, True, 127, 0.0),         # window edges around the tile size
    (777, 4, 4, 64, True, 128, 0.0),
    (900, 8, 1, 128, True, 129, 0.0),
    (2048, 8, 2, 128, True, 1000, 0.0),
    (600, 4, 2, 128, False, 200, 0.0),      # full attention with a left window
    (1000, 8, 2, 128, True, -1, 30.0),      # soft-capping alone
    (700, 4, 2, 64, True, -1, 1.0),         # a tight cap
    (1500, 8, 2, 128, True, 300, 50.0),     # both
    (300, 4, 1, 128, False, -1, 20.0),
    (1000, 8, 4, 256, True, 63, 0.0),        # head_dim 256: 64-key tiles, window edges
    (1000, 8, 4, 256, True, 64, 0.0),
    (700, 4, 2, 256, False, 150, 0.0),
    (900, 8, 4, 256, True, -1, 30.0),
    (1100, 8, 4, 256, True, 200, 50.0),
])
def test_prefill_variants_full(dev, N, Hq, Hkv, D, causal, Wl, cap):
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=N + Wl, causal=causal)
    o, lse = run_prefill(x, dev, window_left=Wl, softcap=cap)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal, window_left=Wl, softcap=cap)
    compare(o, lse, o_ref, lse_ref, f"prefill N={N} W={Wl} cap={cap}")


@pytest.mark.parametrize("Wl,cap", [(4095, 0.0), (-1, 50.0), (4095, 50.0)])
def test_prefill_variants_qwen_8192_sampled(dev, Wl, cap):
    """Qwen2.5-7B layer shape at N = 8192 with a 4096-token window and/or a
    cap of 50: 512 sampled rows, including the window's edges."""
    x = W.qwen_prefill(8192)
    o, lse = run_prefill(x, dev, window_left=Wl, softcap=cap)
    rng = np.random.default_rng(3)
    rows = [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 28, 500), rng.integers(0, 8192, 500))]
    rows += [(0, 0, i) for i in (0, 127, 128, 4095, 4096, 4097, 4223, 4224, 8191, 6000, 5000, 4500)]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, True, rows, window_left=Wl,
                                         softcap=cap)
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    compare(o[idx], lse[idx], o_ref, lse_ref, f"qwen 8192 W={Wl} cap={cap}")


def test_window_covering_everything_equals_plain(dev):
    x = W.make_prefill(1, 8, 2, 1000, 128, seed=5)
    o1, l1 = run_prefill(x, dev)
    o2, l2 = run_prefill(x, dev, window_left=5000)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def run_decode(d, dev, S, Wl, cap):
    q, kc, vc, lens = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    B, Hq, D = q.shape
    op, lp = nan_like((S, B, Hq, D), dev), nan_like((S, B, Hq), dev)
    attn.decode_splitkv(q, kc, vc, lens, bt, num_splits=S, max_kv_len=d.max_kv_len or None,
                        scale=d.scale, o_partial=op, lse_partial=lp, window_left=Wl, softcap=cap)
    o, lse = nan_like((B, Hq, D), dev), nan_like((B, Hq), dev)
    attn.combine(op, lp, out=o, lse=lse)
    attn.check_device_status()
    return op, lp, o, lse


@pytest.mark.parametrize("paged,lens,S,Wl,cap", [
    (False, [3000], 7, 100, 0.0),
    (False, [3000], 7, 0, 0.0),
    (False, [30720], 76, 4095, 0.0),
    (False, [2000], 5, -1, 50.0),
    (False, [2000], 5, 300, 30.0),
    (True, [1000, 17, 5000, 64], 6, 15, 0.0),
    (True, [1000, 17, 5000, 64], 6, 16, 0.0),
    (True, [1000, 17, 5000, 64], 6, 17, 20.0),
    (True, [4097, 1, 300], 3, 4000, 0.0),
])
def test_decode_variants(dev, paged, lens, S, Wl, cap):
    if paged:
        d = W.make_decode_paged(len(lens), 16, 4, 128, lens, block_size=16, seed=sum(lens) + S)
    else:
        d = W.make_decode_contiguous(len(lens), 28, 4, 128, lens[0], seed=lens[0] + Wl)
    op, lp, o, lse = run_decode(d, dev, S, Wl, cap)
    L = d.kv_lens.tolist()
    o_ref, lse_ref = oracle.decode(d.q, d.k_cache, d.v_cache, d.block_table, L, d.scale,
                                   d.block_size, window_left=Wl, softcap=cap)
    compare(o, lse, o_ref, lse_ref, f"decode W={Wl} cap={cap}")
    ranges = [split_ranges(n, S, Wl) for n in L]
    op_ref, lp_ref = oracle.decode_partials(d.q, d.k_cache, d.v_cache, d.block_table, L, d.scale,
                                            d.block_size, ranges, softcap=cap)
    compare(op, lp, op_ref, lp_ref, f"decode partials W={Wl} cap={cap}")


def test_decode_window_equals_last_prefill_row(dev):
    x = W.make_prefill(1, 28, 4, 1500, 128, seed=9)
    o_p, l_p = run_prefill(x, dev, window_left=200, softcap=25.0)
    kc = x.k[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    vc = x.v[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    d = W.DecodeInputs(x.q[:, :, -1].contiguous(), kc, vc, None,
                       torch.tensor([1500], dtype=torch.int32), 0, x.scale, 1500)
    _, _, o_d, l_d = run_decode(d, dev, 4, 200, 25.0)
    assert (o_d - o_p[:, :, -1]).abs().max().item() <= 1e-2
    assert (l_d - l_p[:, :, -1]).abs().max().item() <= 1e-3


def alibi_slopes(n_heads):
    """The usual geometric ALiBi slopes 2^(-8 (h+1) / n_heads)."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / n_heads) for h in range(n_heads)],
                        dtype=torch.float32)


@pytest.mark.parametrize("N,Hq,Hkv,D,causal,Wl", [
    (1000, 8, 2, 128, True, -1),
    (777, 4, 4, 64, True, -1),
    (600, 8, 2, 128, False, -1),
    (1500, 8, 2, 128, True, 300),
    (900, 8, 4, 256, True, -1),              # head_dim 256
    (700, 4, 2, 256, False, 100),
])
def test_prefill_alibi_full(dev, N, Hq, Hkv, D, causal, Wl):
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=N + 7, causal=causal)
    sl = alibi_slopes(Hq)
    o, lse = run_prefill(x, dev, window_left=Wl, alibi_slopes=sl.to(dev))
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal, window_left=Wl,
                                    alibi_slopes=sl.tolist())
    compare(o, lse, o_ref, lse_ref, f"alibi prefill N={N} W={Wl}")


@pytest.mark.parametrize("N,Hq,Hkv,D,causal,Wl,slopes", [
    (700, 4, 2, 64, False, -1, None),        # head_dim 64, tiles on both sides of the diagonal
    (1100, 8, 2, 128, False, 300, None),     # non-causal window: keys on both sides within it
    (640, 8, 4, 128, True, -1, [1.0, 0.9, 0.02, 0.25, 0.5, 0.001, 0.75, 0.33]),
    (640, 8, 4, 128, False, -1, [1.0, -0.05, 0.02, 0.25, 0.5, 0.001, 0.75, 0.0]),
])
def test_prefill_alibi_bias_forms(dev, N, Hq, Hkv, D, causal, Wl, slopes):
    """At head_dim <= 128 the kernel splits -slope |i - j| per key tile into
    a row constant and a per-key part that the tensor core adds (the slope
    carried as three bf16 terms); these cases cover tiles below, above and on
    the diagonal, steep, zero and negative slopes."""
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=N + 11, causal=causal)
    sl = alibi_slopes(Hq) if slopes is None else torch.tensor(slopes, dtype=torch.float32)
    o, lse = run_prefill(x, dev, window_left=Wl, alibi_slopes=sl.to(dev))
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal, window_left=Wl,
                                    alibi_slopes=sl.tolist())
    compare(o, lse, o_ref, lse_ref, f"alibi bias forms N={N} D={D} causal={causal} W={Wl}")


def test_prefill_alibi_qwen_8192_sampled(dev):
    x = W.qwen_prefill(8192)
    sl = alibi_slopes(28)
    o, lse = run_prefill(x, dev, alibi_slopes=sl.to(dev))
    rng = np.random.default_rng(4)
    rows = [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 28, 400), rng.integers(0, 8192, 400))]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, True, rows,
                                         alibi_slopes=sl.tolist())
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    compare(o[idx], lse[idx], o_ref, lse_ref, "alibi qwen 8192")


@pytest.mark.parametrize("paged,lens,S,Wl", [
    (False, [3000], 7, -1), (False, [30720], 76, -1), (False, [2000], 5, 300),
    (True, [1000, 17, 5000, 64], 6, -1), (True, [1000, 17, 5000, 64], 6, 40),
])
def test_decode_alibi(dev, paged, lens, S, Wl):
    if paged:
        d = W.make_decode_paged(len(lens), 16, 4, 128, lens, block_size=16, seed=sum(lens) + 1)
        Hq = 16
    else:
        d = W.make_decode_contiguous(len(lens), 28, 4, 128, lens[0], seed=lens[0] + 2)
        Hq = 28
    sl = alibi_slopes(Hq)
    q, kc, vc, lens_d = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    B = q.shape[0]
    op, lp = nan_like((S, B, Hq, 128), dev), nan_like((S, B, Hq), dev)
    attn.decode_splitkv(q, kc, vc, lens_d, bt, num_splits=S, max_kv_len=d.max_kv_len or None,
                        scale=d.scale, o_partial=op, lse_partial=lp, window_left=Wl,
                        alibi_slopes=sl.to(dev))
    o, lse = attn.combine(op, lp)
    attn.check_device_status()
    L = d.kv_lens.tolist()
    o_ref, lse_ref = oracle.decode(d.q, d.k_cache, d.v_cache, d.block_table, L, d.scale,
                                   d.block_size, window_left=Wl, alibi_slopes=sl.tolist())
    compare(o, lse, o_ref, lse_ref, f"alibi decode W={Wl}")
    ranges = [split_ranges(n, S, Wl) for n in L]
    op_ref, lp_ref = oracle.decode_partials(d.q, d.k_cache, d.v_cache, d.block_table, L, d.scale,
                                            d.block_size, ranges, alibi_slopes=sl.tolist())
    # far splits carry biases of -slope * distance ~ -2.5e4: their fp32 LSE
    # is only good to a few units in the last place of that magnitude
    compare(op, lp, op_ref, lp_ref, f"alibi decode partials W={Wl}", lse_rel=2.0 ** -21)


@pytest.mark.parametrize("D,paged,lens,S,Wl,cap,alibi", [
    (64, True, [1000, 17, 3000], 5, 100, 0.0, False),      # head_dim 64: window
    (64, False, [2500], 6, -1, 30.0, False),                # soft-capping
    (64, True, [700, 2000], 4, -1, 0.0, True),              # ALiBi
    (256, True, [1000, 17, 3000], 5, 200, 0.0, False),     # head_dim 256: window
    (256, False, [2500], 6, 64, 50.0, False),               # window + soft-capping
    (256, True, [700, 2000], 4, 300, 0.0, True),            # ALiBi with a window
])
def test_decode_variants_other_head_dims(dev, D, paged, lens, S, Wl, cap, alibi):
    """Decode variants at head_dim 64 and 256 (the combined result)."""
    _decode_variant_case(dev, D, paged, lens, S, Wl, cap, alibi, 8, 4 if paged else 2)


@pytest.mark.parametrize("D,paged,lens,S,Wl,cap,alibi,Hq,Hkv", [
    (128, True, [1700, 40], 6, -1, 0.0, True, 64, 2),      # ALiBi, g = 32
    (128, False, [3000], 7, 500, 40.0, False, 64, 1),      # window + cap, g = 64
    (256, True, [900, 2100], 3, 100, 0.0, False, 48, 1),   # window, g = 48, head_dim 256
])
def test_decode_variants_large_gqa(dev, D, paged, lens, S, Wl, cap, alibi, Hq, Hkv):
    """Decode variants with more than 16 query heads per kv head."""
    _decode_variant_case(dev, D, paged, lens, S, Wl, cap, alibi, Hq, Hkv)


def _decode_variant_case(dev, D, paged, lens, S, Wl, cap, alibi, Hq, Hkv):
    if paged:
        d = W.make_decode_paged(len(lens), Hq, Hkv, D, lens, block_size=16, seed=sum(lens) + D)
    else:
        d = W.make_decode_contiguous(len(lens), Hq, Hkv, D, lens[0], seed=lens[0] + D)
    sl = alibi_slopes(Hq) if alibi else None
    q, kc, vc, ln = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    o, lse = attn.decode(q, kc, vc, ln, bt, num_splits=S, max_kv_len=d.max_kv_len or None,
                         scale=d.scale, window_left=Wl, softcap=cap,
                         alibi_slopes=sl.to(dev) if alibi else None)
    attn.check_device_status()
    o_ref, lse_ref = oracle.decode(d.q, d.k_cache, d.v_cache, d.block_table, d.kv_lens.tolist(),
                                   d.scale, d.block_size, window_left=Wl, softcap=cap,
                                   alibi_slopes=sl.tolist() if alibi else None)
    compare(o, lse, o_ref, lse_ref, f"decode d={D} W={Wl} cap={cap} alibi={alibi}")
