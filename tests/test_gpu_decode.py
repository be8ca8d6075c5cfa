"""Parity of split-KV decode (attn_decode_splitkv) and the combine
(attn_combine), through the C ABI, against the float64 oracle: the combined
result and every split's partial result, contiguous and paged caches, the
split-count sweep, edge cases, and the kernels' own error reporting."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
from exact_io_aware_order_gb300._lib import AttnError, status_codes
import oracle
from gpu_util import compare, nan_like

pytestmark = pytest.mark.gpu


def split_rule(kv_len, S):
    """The header's split rule, restated here: c = roundup(ceil(len/S), 16)."""
    if kv_len == 0:
        return [(0, 0)] * S
    c = ((kv_len + S - 1) // S + 15) // 16 * 16
    return [(min(s * c, kv_len), min(min(s * c, kv_len) + c, kv_len)) for s in range(S)]


def run_decode(d, dev, S):
    q = d.q.to(dev)
    kc, vc = d.k_cache.to(dev), d.v_cache.to(dev)
    lens = d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    B, Hq, D = q.shape
    op, lp = nan_like((S, B, Hq, D), dev), nan_like((S, B, Hq), dev)
    attn.decode_splitkv(q, kc, vc, lens, bt, num_splits=S, max_kv_len=d.max_kv_len, scale=d.scale,
                        o_partial=op, lse_partial=lp)
    o, lse = nan_like((B, Hq, D), dev), nan_like((B, Hq), dev)
    attn.combine(op, lp, out=o, lse=lse)
    attn.check_device_status()
    return op, lp, o, lse


def check_all(d, op, lp, o, lse, S, what):
    bt = d.block_table
    lens = d.kv_lens.tolist()
    o_ref, lse_ref = oracle.decode(d.q, d.k_cache, d.v_cache, bt, lens, d.scale, d.block_size)
    res = compare(o, lse, o_ref, lse_ref, what + " combined")
    ranges = [split_rule(n, S) for n in lens]
    op_ref, lp_ref = oracle.decode_partials(d.q, d.k_cache, d.v_cache, bt, lens, d.scale,
                                            d.block_size, ranges)
    compare(op, lp, op_ref, lp_ref, what + " partials")
    return res


@pytest.mark.parametrize("S", [1, 16, 64, 148])
def test_qwen_decode_split_sweep(dev, S):
    """28 / 4 heads, head_dim 128, contiguous 30720-token cache."""
    d = W.qwen_decode(30720)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"qwen S={S}")


def test_paged_batched_decode_auto_splits(dev):
    """16 sequences, lengths uniform in [1024, 32768], 32 / 8 heads, 16-token blocks."""
    d = W.llama_paged_decode()
    S = attn.decode_num_splits(16, 8, d.max_kv_len)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"paged S={S}")


@pytest.mark.parametrize("lens,S,bs,D,Hq,Hkv", [
    ([0, 1, 15, 16, 17], 3, 16, 128, 8, 2),
    ([63, 64, 65, 200], 2, 16, 64, 4, 4),
    ([5, 1000], 100, 16, 128, 16, 1),        # many empty splits, g = 16
    ([1, 2, 3], 1, 1, 128, 2, 1),            # one-token blocks
    ([777, 1], 5, 7, 64, 6, 3),              # odd block size
    ([4096], 1, 64, 128, 28, 4),
    ([0, 1, 15, 16, 17, 3000], 4, 16, 256, 16, 8),   # head_dim 256, 16-token boxes
    ([777, 1], 5, 7, 256, 4, 2),                     # head_dim 256, plain loads
])
def test_paged_edge_cases(dev, lens, S, bs, D, Hq, Hkv):
    d = W.make_decode_paged(len(lens), Hq, Hkv, D, lens, block_size=bs, seed=sum(lens) + S,
                            extra_blocks=3)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"paged lens={lens} S={S}")


@pytest.mark.parametrize("kv_len,L,S", [(1, 1, 1), (100, 300, 4), (30720, 30720, 7),
                                        (2049, 4096, 33)])
def test_contiguous_edge_cases(dev, kv_len, L, S):
    d = W.make_decode_contiguous(2, 8, 2, 128, kv_len, seed=kv_len, max_kv_len=L)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"contig len={kv_len} L={L} S={S}")


@pytest.mark.parametrize("paged", [False, True])
def test_long_cache_262144(dev, paged):
    """One sequence of 262144 cached tokens (8 / 2 heads; 16384 blocks when
    paged), the policy's split count: every split's partials and the
    combined result against the oracle."""
    L = 262144
    d = (W.make_decode_paged(1, 8, 2, 128, [L], seed=21) if paged
         else W.make_decode_contiguous(1, 8, 2, 128, L, seed=21))
    S = attn.decode_num_splits(1, 2, L)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"len={L} paged={paged} S={S}")


@pytest.mark.parametrize("kv_len,L,S", [(1, 1, 1), (4100, 4200, 5), (30720, 30720, 60)])
def test_contiguous_head_dim_256(dev, kv_len, L, S):
    """head_dim 256 (four 128-byte swizzle spans per cached row), 16 / 8 heads."""
    d = W.make_decode_contiguous(2, 16, 8, 256, kv_len, seed=kv_len + 256, max_kv_len=L)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"contig d256 len={kv_len} L={L} S={S}")


def test_slots_past_the_end_are_never_read(dev):
    """NaN in cache slots beyond kv_len (paged tail and contiguous tail) must not
    reach the output."""
    d = W.make_decode_paged(2, 8, 2, 128, [37, 50], block_size=16, seed=3)
    for b, n in enumerate(d.kv_lens.tolist()):
        last = int(d.block_table[b, (n - 1) // 16])
        d.k_cache[last, n % 16 or 16:] = float("nan")
        d.v_cache[last, n % 16 or 16:] = float("nan")
    op, lp, o, lse = run_decode(d, dev, 3)
    check_all(d, op, lp, o, lse, 3, "nan tail paged")
    c = W.make_decode_contiguous(1, 4, 1, 64, 90, seed=4, max_kv_len=200)
    c.k_cache[:, 90:] = float("nan")
    c.v_cache[:, 90:] = float("nan")
    op, lp, o, lse = run_decode(c, dev, 2)
    check_all(c, op, lp, o, lse, 2, "nan tail contiguous")


def test_split_count_does_not_change_the_result(dev):
    d = W.make_decode_contiguous(1, 28, 4, 128, 5000, seed=6)
    outs = [run_decode(d, dev, S)[2:] for S in (1, 3, 64, 300)]
    for o, lse in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= 2e-3
        assert (lse - outs[0][1]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("Hq,Hkv,D", [(28, 4, 128), (16, 8, 256)])
def test_decode_matches_last_prefill_row(dev, Hq, Hkv, D):
    x = W.make_prefill(1, Hq, Hkv, 1111, D, seed=8)
    o_p, lse_p = attn.prefill(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.scale, True)
    kc = x.k[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    vc = x.v[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    d = W.DecodeInputs(x.q[:, :, -1].contiguous(), kc, vc, None,
                       torch.tensor([1111], dtype=torch.int32), 0, x.scale, 1111)
    _, _, o_d, lse_d = run_decode(d, dev, 9)
    assert (o_d - o_p[:, :, -1]).abs().max().item() <= 1e-2
    assert (lse_d - lse_p[:, :, -1]).abs().max().item() <= 1e-3


def test_combine_kernel_on_arbitrary_partials(dev):
    rng = np.random.default_rng(0)
    for S, B, Hq, D in [(5, 2, 3, 128), (148, 1, 28, 128), (1, 4, 2, 64), (1024, 1, 2, 64),
                        (1024, 1, 1, 64), (7, 2, 3, 256), (300, 1, 16, 256)]:
        op = rng.standard_normal((S, B, Hq, D)).astype(np.float32)
        lp = (rng.standard_normal((S, B, Hq)) * 5).astype(np.float32)
        lp[rng.random((S, B, Hq)) < 0.2] = -np.inf            # empty splits
        lp[:, 0, 0] = -np.inf                                 # one row with every split empty
        op[np.isneginf(lp)] = 0.0
        o, lse = attn.combine(torch.from_numpy(op).to(dev), torch.from_numpy(lp).to(dev))
        attn.check_device_status()
        o_ref, lse_ref = oracle.combine(op.astype(np.float64), lp.astype(np.float64))
        ol, ll = o.double().cpu().numpy(), lse.double().cpu().numpy()
        assert np.array_equal(np.isneginf(ll), np.isneginf(lse_ref))
        fin = np.isfinite(lse_ref)
        if fin.any():
            assert np.abs(ll[fin] - lse_ref[fin]).max() <= 1e-5
        assert np.abs(ol - o_ref).max() <= 1e-5
        assert np.all(ol[~fin] == 0.0)


def test_bad_block_table_entry_is_reported(dev):
    """An out-of-range physical block id is caught by the kernel's own bounds
    check (the copy is redirected to block 0) and reported as ATTN_ERR_DEVICE."""
    d = W.make_decode_paged(1, 4, 1, 128, [40], block_size=16, seed=1)
    d.block_table[0, 1] = d.k_cache.shape[0] + 5
    with pytest.raises(AttnError) as e:
        run_decode(d, dev, 2)
    assert e.value.status == status_codes()["ATTN_ERR_DEVICE"]
    attn.check_device_status()                                  # the word was cleared


def test_kv_len_beyond_capacity_is_reported(dev):
    d = W.make_decode_contiguous(1, 4, 1, 128, 64, seed=2)
    d.kv_lens[0] = 65                                           # capacity is 64
    with pytest.raises(AttnError) as e:
        run_decode(d, dev, 2)
    assert e.value.status == status_codes()["ATTN_ERR_DEVICE"]
    attn.check_device_status()


def test_bounded_wait_gives_up_and_reports(dev):
    """A kernel waiting on a barrier nobody arrives at returns after the
    timeout with ATTN_ERR_TIMEOUT; the context stays usable."""
    old = attn.set_wait_timeout_ns(2_000_000)                    # 2 ms
    try:
        assert attn.selftest_bounded_wait() == status_codes()["ATTN_ERR_TIMEOUT"]
    finally:
        attn.set_wait_timeout_ns(old)
    d = W.make_decode_contiguous(1, 4, 2, 128, 300, seed=3)
    op, lp, o, lse = run_decode(d, dev, 2)
    check_all(d, op, lp, o, lse, 2, "after timeout test")


@pytest.mark.parametrize("Hq,Hkv,D,lens,S,bs", [
    (32, 1, 128, [3000], 8, 16),          # g = 32 (multi-query-like)
    (64, 1, 128, [2500, 17], 5, 16),      # g = 64
    (40, 2, 64, [1000, 0, 33], 3, 16),    # g = 20: a partly filled second row group
    (96, 2, 256, [1500], 4, 16),          # g = 48, head_dim 256
    (64, 2, 128, [700, 1], 7, 7),         # g = 32, odd block size (plain loads)
])
def test_large_gqa_ratio_paged(dev, Hq, Hkv, D, lens, S, bs):
    """Query heads per kv head above 16: the warps split into row groups of 16
    rows; every K/V row is still read once (page "FlashAttention for
    inference", section "Decode: a different bottleneck", GQA paragraph)."""
    d = W.make_decode_paged(len(lens), Hq, Hkv, D, lens, block_size=bs, seed=Hq + D + S,
                            extra_blocks=2)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"paged g={Hq // Hkv} D={D} lens={lens}")


@pytest.mark.parametrize("Hq,Hkv,kv_len,S", [(64, 1, 30720, 76), (32, 1, 5000, 19), (48, 1, 777, 3)])
def test_large_gqa_ratio_contiguous(dev, Hq, Hkv, kv_len, S):
    d = W.make_decode_contiguous(1, Hq, Hkv, 128, kv_len, seed=kv_len + Hq)
    op, lp, o, lse = run_decode(d, dev, S)
    check_all(d, op, lp, o, lse, S, f"contig g={Hq // Hkv} len={kv_len}")


def test_gqa_ratio_above_64_is_refused(dev):
    d = W.make_decode_contiguous(1, 65, 1, 64, 32, seed=1)
    with pytest.raises(AttnError) as e:
        run_decode(d, dev, 1)
    assert e.value.status == status_codes()["ATTN_ERR_GQA"]


@pytest.mark.parametrize("paged", [False, True])
def test_early_cache_chain(dev, paged):
    """Layers chained on one stream, each decode (ATTN_DECODE_EARLY_CACHE)
    right after the previous layer's combine, each layer with its own cache
    and query (so the previous kernel writes none of what the decode reads
    early): every layer's combined result against the oracle, and equal, bit
    for bit, to the same decode without the flag."""
    layers = 3
    if paged:
        ds = [W.make_decode_paged(3, 8, 2, 128, [3000, 17, 1024], block_size=16, seed=40 + i)
              for i in range(layers)]
    else:
        ds = [W.make_decode_contiguous(2, 8, 2, 128, 3000, seed=40 + i, max_kv_len=3100)
              for i in range(layers)]
    S = 7
    dev_in = []
    for d in ds:
        dev_in.append((d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev),
                       d.block_table.to(dev) if d.block_table is not None else None))
    B, Hq, D = ds[0].q.shape
    op = torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev)
    lp = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
    outs = {}
    for early in (True, False):
        res = []
        for i, d in enumerate(ds):
            q, kc, vc, lens, bt = dev_in[i]
            attn.decode_splitkv(q, kc, vc, lens, bt, num_splits=S, max_kv_len=d.max_kv_len,
                                scale=d.scale, o_partial=op, lse_partial=lp, early_cache=early)
            o, lse = nan_like((B, Hq, D), dev), nan_like((B, Hq), dev)
            attn.combine(op, lp, out=o, lse=lse)
            res.append((o, lse))
        torch.cuda.synchronize()
        attn.check_device_status()
        outs[early] = res
    for i, d in enumerate(ds):
        o, lse = outs[True][i]
        o_ref, lse_ref = oracle.decode(d.q, d.k_cache, d.v_cache, d.block_table,
                                       d.kv_lens.tolist(), d.scale, d.block_size)
        compare(o, lse, o_ref, lse_ref, f"early chain layer {i} paged={paged}")
        assert torch.equal(o, outs[False][i][0]) and torch.equal(lse, outs[False][i][1])


def test_early_cache_refused_with_append(dev):
    """The appending decode writes the cache itself: no early streaming there
    (the C entry points that append take no flags; the binding has none)."""
    import inspect
    assert "early_cache" not in inspect.signature(attn.decode_append_splitkv).parameters


@pytest.mark.parametrize("paged,D,Hq,Hkv,variant", [
    (True, 128, 8, 2, {"window_left": 200}),
    (False, 128, 8, 2, {"alibi": True}),
    (True, 256, 4, 2, {"softcap": 30.0}),
    (False, 64, 4, 4, {}),
    (True, 128, 32, 1, {}),                    # 32 query heads per kv head (row-group teams)
])
def test_early_cache_chain_variants(dev, paged, D, Hq, Hkv, variant):
    """Early cache streaming with the decode variants, head_dims and GQA
    ratios: two chained layers equal, bit for bit, the same decodes without
    the flag, and match the oracle."""
    import oracle as O
    kw = {k: v for k, v in variant.items() if k != "alibi"}
    okw = dict(kw)
    if variant.get("alibi"):
        sl = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)
        kw["alibi_slopes"] = sl.to(dev)
        okw["alibi_slopes"] = sl.tolist()
    if paged:
        ds = [W.make_decode_paged(2, Hq, Hkv, D, [900, 33], block_size=16, seed=60 + i)
              for i in range(2)]
    else:
        ds = [W.make_decode_contiguous(2, Hq, Hkv, D, 700, seed=60 + i) for i in range(2)]
    S = 5
    B = ds[0].q.shape[0]
    outs = {}
    for early in (True, False):
        res = []
        for d in ds:
            op = torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev)
            lp = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
            bt = d.block_table.to(dev) if d.block_table is not None else None
            attn.decode_splitkv(d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev),
                                d.kv_lens.to(dev), bt, num_splits=S, max_kv_len=d.max_kv_len,
                                scale=d.scale, o_partial=op, lse_partial=lp, early_cache=early,
                                **kw)
            res.append(attn.combine(op, lp))
        torch.cuda.synchronize()
        attn.check_device_status()
        outs[early] = res
    for i, d in enumerate(ds):
        o, lse = outs[True][i]
        assert torch.equal(o, outs[False][i][0]) and torch.equal(lse, outs[False][i][1])
        o_ref, lse_ref = O.decode(d.q, d.k_cache, d.v_cache, d.block_table, d.kv_lens.tolist(),
                                  d.scale, d.block_size, **okw)
        compare(o, lse, o_ref, lse_ref, f"early variants {variant} paged={paged} D={D}")
