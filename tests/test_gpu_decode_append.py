"""Parity of decode with in-place append (attn_decode_append_splitkv), through
the C ABI, against the float64 oracle's decode_append: the combined result,
every split's partial, and the caches afterwards (bit for bit: the new rows
are written at position kv_lens[b], nothing else changes)."""

import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
from exact_io_aware_order_gb300._lib import AttnError, status_codes
import oracle
from gpu_util import compare, nan_like

pytestmark = pytest.mark.gpu


def split_rule(kv_len, S):
    """The header's split rule: c = roundup(ceil(len/S), 16)."""
    if kv_len == 0:
        return [(0, 0)] * S
    c = ((kv_len + S - 1) // S + 15) // 16 * 16
    return [(min(s * c, kv_len), min(min(s * c, kv_len) + c, kv_len)) for s in range(S)]


def new_rows(B, n_kv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, n_kv, d, generator=g).to(torch.bfloat16),
            torch.randn(B, n_kv, d, generator=g).to(torch.bfloat16))


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


def run_append(d, kn, vn, dev, S):
    q, kc, vc, lens = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    B, Hq, D = q.shape
    op, lp = nan_like((S, B, Hq, D), dev), nan_like((S, B, Hq), dev)
    attn.decode_append_splitkv(q, kn.to(dev), vn.to(dev), kc, vc, lens, bt, num_splits=S,
                               max_kv_len=d.max_kv_len or None, scale=d.scale, o_partial=op,
                               lse_partial=lp)
    o, lse = nan_like((B, Hq, D), dev), nan_like((B, Hq), dev)
    attn.combine(op, lp, out=o, lse=lse)
    attn.check_device_status()
    assert torch.equal(lens.cpu(), d.kv_lens)              # lengths are the caller's to bump
    return op, lp, o, lse, kc, vc


def check_append(d, kn, vn, dev, S, what):
    op, lp, o, lse, kc, vc = run_append(d, kn, vn, dev, S)
    lens = d.kv_lens.tolist()
    o_ref, lse_ref, kc_ref, vc_ref = oracle.decode_append(d.q, kn, vn, d.k_cache, d.v_cache,
                                                          d.block_table, lens, d.scale,
                                                          d.block_size)
    compare(o, lse, o_ref, lse_ref, what + " combined")
    ranges = [split_rule(n + 1, S) for n in lens]
    op_ref, lp_ref = oracle.decode_partials(d.q, kc_ref, vc_ref, d.block_table,
                                            [n + 1 for n in lens], d.scale, d.block_size, ranges)
    compare(op, lp, op_ref, lp_ref, what + " partials")
    assert torch.equal(bits(kc), bits(kc_ref)), what + ": K cache differs from the appended one"
    assert torch.equal(bits(vc), bits(vc_ref)), what + ": V cache differs from the appended one"


def paged_with_room(B, Hq, Hkv, D, lens, bs, seed):
    """A paged cache holding lens[b] tokens with a slot allocated for one more
    (the slot holds stale data the append overwrites); tails past it are NaN."""
    d = W.make_decode_paged(B, Hq, Hkv, D, [n + 1 for n in lens], block_size=bs, seed=seed,
                            extra_blocks=2)
    d.kv_lens = torch.as_tensor(lens, dtype=torch.int32)
    for b, n in enumerate(lens):
        blk = int(d.block_table[b, n // bs])
        d.k_cache[blk, n % bs + 1:] = float("nan")
        d.v_cache[blk, n % bs + 1:] = float("nan")
    return d


@pytest.mark.parametrize("lens,S,bs,D,Hq,Hkv", [
    ([0, 1, 15, 16, 31], 3, 16, 128, 8, 2),     # empty cache, block boundaries
    ([63, 64, 200], 2, 16, 64, 4, 4),
    ([5, 1000], 100, 16, 128, 16, 1),           # many empty splits, g = 16
    ([0, 2, 3], 1, 1, 128, 2, 1),               # one-token blocks
    ([776, 0], 5, 7, 64, 6, 3),                 # odd block size (plain-load path)
    ([4095], 7, 64, 128, 28, 4),
    ([0, 31, 2000], 4, 16, 256, 16, 8),         # head_dim 256
    ([40, 0], 3, 7, 256, 4, 2),                 # head_dim 256, plain loads
    ([0, 33, 1500], 4, 16, 128, 64, 1),         # g = 64: four row groups
])
def test_paged_append(dev, lens, S, bs, D, Hq, Hkv):
    d = paged_with_room(len(lens), Hq, Hkv, D, lens, bs, seed=sum(lens) + S)
    kn, vn = new_rows(len(lens), Hkv, D, seed=S)
    check_append(d, kn, vn, dev, S, f"paged append lens={lens} S={S} bs={bs}")


@pytest.mark.parametrize("kv_len,L,S", [(0, 1, 1), (0, 64, 3), (99, 300, 4), (30719, 30720, 76),
                                        (2048, 4096, 33)])
def test_contiguous_append(dev, kv_len, L, S):
    d = W.make_decode_contiguous(2, 28, 4, 128, kv_len, seed=kv_len + 1, max_kv_len=L)
    d.k_cache[:, kv_len + 1:] = float("nan")
    d.v_cache[:, kv_len + 1:] = float("nan")
    kn, vn = new_rows(2, 4, 128, seed=kv_len)
    check_append(d, kn, vn, dev, S, f"contiguous append len={kv_len} L={L} S={S}")


def test_token_by_token_reproduces_prefill(dev):
    """Starting from an empty cache full of NaN, appending tokens 0..N-1 one
    decode at a time gives every row of causal prefill of the same sequence,
    and leaves exactly the sequence's keys and values in the cache."""
    N, Hq, Hkv, D, bs = 150, 8, 2, 128, 16
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=21)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    nb = (N + bs - 1) // bs
    perm = torch.randperm(nb + 3, generator=torch.Generator().manual_seed(4))
    table = perm[:nb].to(torch.int32).reshape(1, nb).to(dev)
    kc = torch.full((nb + 3, bs, Hkv, D), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = kc.clone()
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    outs, lses = [], []
    for t in range(N):
        lens = torch.tensor([t], dtype=torch.int32, device=dev)
        o, lse = attn.decode_append(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                    v[:, :, t].contiguous(), kc, vc, lens, table, num_splits=3,
                                    scale=x.scale)
        outs.append(o)
        lses.append(lse)
    attn.check_device_status()
    o_all = torch.stack(outs, dim=2)       # (1, Hq, N, D)
    lse_all = torch.stack(lses, dim=2)     # (1, Hq, N)
    compare(o_all, lse_all, o_ref, lse_ref, "token-by-token append")
    for t in range(N):
        blk, slot = int(perm[t // bs]), t % bs
        assert torch.equal(bits(kc[blk, slot]), bits(x.k[0, :, t]))
        assert torch.equal(bits(vc[blk, slot]), bits(x.v[0, :, t]))


def test_full_cache_is_reported_and_not_written(dev):
    d = W.make_decode_contiguous(1, 4, 1, 128, 64, seed=2)      # capacity 64, all used
    kn, vn = new_rows(1, 1, 128, seed=1)
    kc, vc = d.k_cache.to(dev), d.v_cache.to(dev)
    k0, v0 = kc.clone(), vc.clone()
    with pytest.raises(AttnError) as e:
        attn.decode_append_splitkv(d.q.to(dev), kn.to(dev), vn.to(dev), kc, vc,
                                   d.kv_lens.to(dev), None, num_splits=2, scale=d.scale)
        attn.check_device_status()
    assert e.value.status == status_codes()["ATTN_ERR_DEVICE"]
    assert torch.equal(bits(kc), bits(k0)) and torch.equal(bits(vc), bits(v0))


def test_bad_block_for_new_position_is_reported_and_not_written(dev):
    d = paged_with_room(1, 4, 1, 128, [32], 16, seed=3)
    d.block_table[0, 2] = d.k_cache.shape[0] + 7            # the block of position 32
    kn, vn = new_rows(1, 1, 128, seed=2)
    kc, vc = d.k_cache.to(dev), d.v_cache.to(dev)
    k0, v0 = kc.clone(), vc.clone()
    with pytest.raises(AttnError) as e:
        attn.decode_append_splitkv(d.q.to(dev), kn.to(dev), vn.to(dev), kc, vc,
                                   d.kv_lens.to(dev), d.block_table.to(dev), num_splits=2,
                                   scale=d.scale)
        attn.check_device_status()
    assert e.value.status == status_codes()["ATTN_ERR_DEVICE"]
    assert torch.equal(bits(kc), bits(k0)) and torch.equal(bits(vc), bits(v0))


def _alibi(n_heads):
    """The usual geometric ALiBi slopes 2^(-8 (h+1) / n_heads)."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / n_heads) for h in range(n_heads)],
                        dtype=torch.float32)


@pytest.mark.parametrize("paged,lens,S,bs,D,Hq,Hkv,Wl,cap,alibi", [
    (True, [0, 31, 2000], 4, 16, 128, 16, 4, 100, 0.0, False),    # window inside the splits
    (False, [30719], 76, 0, 128, 28, 4, 4095, 0.0, False),         # window, full cache
    (True, [5, 1000], 3, 16, 128, 8, 2, -1, 30.0, False),          # soft-capping
    (True, [77, 1500], 5, 7, 128, 8, 2, 64, 50.0, False),          # window + cap, plain loads
    (False, [2048], 33, 0, 128, 8, 2, -1, 0.0, True),              # ALiBi
    (True, [0, 700], 4, 16, 256, 16, 8, 255, 0.0, False),          # head_dim 256 with a window
    (True, [10, 900], 3, 16, 128, 32, 1, -1, 0.0, True),           # ALiBi, g = 32
    (False, [1200], 5, 0, 64, 96, 2, 300, 20.0, False),            # window + cap, g = 48
])
def test_append_with_variants(dev, paged, lens, S, bs, D, Hq, Hkv, Wl, cap, alibi):
    """Decode with append and a sliding window, soft-capping or ALiBi
    (attn_decode_append_splitkv_ex): the combined result against the oracle's
    decode with append under the same variant, and the caches bit for bit."""
    if paged:
        d = paged_with_room(len(lens), Hq, Hkv, D, lens, bs, seed=sum(lens) + S + 17)
    else:
        d = W.make_decode_contiguous(len(lens), Hq, Hkv, D, lens[0], seed=lens[0] + 23,
                                     max_kv_len=lens[0] + 1)
    kn, vn = new_rows(len(lens), Hkv, D, seed=S + 5)
    sl = _alibi(Hq) if alibi else None
    q, kc, vc, ln = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev), d.kv_lens.to(dev)
    bt = d.block_table.to(dev) if d.block_table is not None else None
    o, lse = attn.decode_append(q, kn.to(dev), vn.to(dev), kc, vc, ln, bt, num_splits=S,
                                max_kv_len=d.max_kv_len or None, scale=d.scale, window_left=Wl,
                                softcap=cap, alibi_slopes=sl.to(dev) if alibi else None)
    attn.check_device_status()
    o_ref, lse_ref, kc_ref, vc_ref = oracle.decode_append(
        d.q, kn, vn, d.k_cache, d.v_cache, d.block_table, d.kv_lens.tolist(), d.scale,
        d.block_size, window_left=Wl, softcap=cap, alibi_slopes=sl.tolist() if alibi else None)
    compare(o, lse, o_ref, lse_ref, f"append lens={lens} W={Wl} cap={cap} alibi={alibi}")
    assert torch.equal(bits(kc), bits(kc_ref)) and torch.equal(bits(vc), bits(vc_ref))
