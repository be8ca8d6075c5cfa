"""Parity of the packed variable-length prefill (attn_prefill_varlen), through
the C ABI, against the float64 oracle's prefill_varlen: whole outputs at small
sizes, sampled rows at a 16-prompt batch, rows outside every sequence left
untouched, one packed sequence equal to the padded prefill bit for bit, and
bad cu_seqlens reported."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
from exact_io_aware_order_gb300._lib import AttnError, status_codes
import oracle
from gpu_util import compare, nan_like

pytestmark = pytest.mark.gpu


def run(x, dev):
    n_q, T, d = x.q.shape
    o, lse = nan_like((n_q, T, d), dev), nan_like((n_q, T), dev)
    attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev), x.scale,
                        x.causal, out=o, lse=lse)
    attn.check_device_status()
    return o, lse


@pytest.mark.parametrize("lens,hq,hkv,d,causal,extra", [
    ([1, 127, 128, 129, 300], 8, 2, 128, True, 0),      # tile edges around 128
    ([1000, 7, 256, 0, 513], 28, 4, 128, True, 5),      # an empty sequence, rows past the end
    ([200, 1, 64, 129], 4, 4, 64, True, 3),             # head_dim 64, MHA
    ([130, 300, 5], 8, 1, 128, False, 2),               # full (non-causal) attention per sequence
    ([77], 6, 3, 128, True, 0),                         # a single short sequence
    ([1, 63, 64, 65, 700, 0, 129], 8, 4, 256, True, 4),  # head_dim 256: 64-key tiles
    ([300, 90], 4, 2, 256, False, 0),
])
def test_varlen_full(dev, lens, hq, hkv, d, causal, extra):
    x = W.make_prefill_varlen(lens, hq, hkv, d, seed=sum(lens), extra_rows=extra, causal=causal)
    o, lse = run(x, dev)
    o_ref, lse_ref = oracle.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, x.scale, causal)
    T0 = int(x.cu_seqlens[-1])
    compare(o[:, :T0], lse[:, :T0], o_ref[:, :T0], lse_ref[:, :T0], f"varlen {lens}")
    assert torch.isnan(o[:, T0:]).all() and torch.isnan(lse[:, T0:]).all(), \
        "rows outside every sequence were written"


def test_varlen_sixteen_prompts_sampled(dev):
    """16 prompts, lengths uniform in [256, 4096], 28 / 4 heads: every
    sequence's first, last and boundary-adjacent rows plus random rows."""
    x = W.qwen_varlen_prefill()
    o, lse = run(x, dev)
    cu = x.cu_seqlens.tolist()
    rng = np.random.default_rng(0)
    rows = []
    for a, b in zip(cu[:-1], cu[1:]):
        for i in {a, a + 1, a + 127, a + 128, b - 1, b - 2} | set(rng.integers(a, b, 4).tolist()):
            if a <= i < b:
                rows.append((int(rng.integers(0, 28)), int(i)))
    o_ref, lse_ref = oracle.prefill_varlen_rows(x.q, x.k, x.v, cu, x.scale, True, rows)
    hs = torch.tensor([h for h, _ in rows])
    ix = torch.tensor([i for _, i in rows])
    compare(o[hs, ix], lse[hs, ix], o_ref, lse_ref, "16 prompts sampled")


def test_one_sequence_equals_padded_prefill_bitwise(dev):
    """One packed sequence is exactly the padded batch-1 prefill: same tiles,
    same arithmetic, so the same bits."""
    x = W.make_prefill(1, 28, 4, 1500, 128, seed=3)
    o_p, l_p = attn.prefill(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.scale, True)
    cu = torch.tensor([0, 1500], dtype=torch.int32, device=dev)
    o_v, l_v = attn.prefill_varlen(x.q[0].to(dev), x.k[0].to(dev), x.v[0].to(dev), cu, x.scale, True)
    attn.check_device_status()
    assert torch.equal(o_v, o_p[0]) and torch.equal(l_v, l_p[0])


def test_bad_cu_seqlens_is_reported(dev):
    x = W.make_prefill_varlen([100, 100], 4, 2, 64, seed=1)
    cu = torch.tensor([0, 150, 120], dtype=torch.int32, device=dev)   # decreasing
    with pytest.raises(AttnError) as e:
        attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), cu, x.scale, True)
        attn.check_device_status()
    assert e.value.status == status_codes()["ATTN_ERR_DEVICE"]
    attn.check_device_status()                                          # cleared


def _slopes(n):
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / n) for h in range(n)], dtype=torch.float32)


@pytest.mark.parametrize("lens,hq,hkv,d,causal,variant", [
    ([300, 0, 129, 1000, 7], 8, 2, 128, True, {"window_left": 100}),
    ([300, 0, 129, 1000, 7], 8, 2, 128, False, {"window_left": 200}),
    ([513, 64, 200], 4, 2, 64, True, {"softcap": 30.0}),
    ([513, 64, 200], 4, 2, 128, False, {"softcap": 20.0, "window_left": 150}),
    ([700, 90, 33], 8, 4, 128, True, {"alibi": True}),
    ([700, 90, 33], 8, 4, 128, False, {"alibi": True}),
    ([400, 129], 4, 2, 256, True, {"alibi": True, "window_left": 90}),
    ([400, 129, 1], 4, 2, 64, False, {"alibi": True}),
])
def test_varlen_variants(dev, lens, hq, hkv, d, causal, variant):
    """Packed prefill with a sliding window, soft-capping or ALiBi
    (``attn_prefill_varlen_ex``): every sequence on its own rows, positions
    from its first row, against the oracle."""
    x = W.make_prefill_varlen(lens, hq, hkv, d, seed=sum(lens) + d, extra_rows=2, causal=causal)
    kw = {k: v for k, v in variant.items() if k != "alibi"}
    okw = dict(kw)
    if variant.get("alibi"):
        sl = _slopes(hq)
        kw["alibi_slopes"] = sl.to(dev)
        okw["alibi_slopes"] = sl.tolist()
    n_q, T, dd = x.q.shape
    o, lse = nan_like((n_q, T, dd), dev), nan_like((n_q, T), dev)
    attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev), x.scale,
                        causal, out=o, lse=lse, **kw)
    attn.check_device_status()
    o_ref, lse_ref = oracle.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, x.scale, causal, **okw)
    T0 = int(x.cu_seqlens[-1])
    compare(o[:, :T0], lse[:, :T0], o_ref[:, :T0], lse_ref[:, :T0], f"varlen {lens} {variant}")
    assert torch.isnan(o[:, T0:]).all() and torch.isnan(lse[:, T0:]).all()


@pytest.mark.parametrize("n_seqs,d,variant", [(1100, 64, {}), (1030, 128, {"window_left": 20}),
                                              (700, 64, {"alibi": True})])
def test_more_sequences_than_one_launch(dev, n_seqs, d, variant):
    """More than 512 packed sequences (lengths 0 .. 48, some empty): the call
    runs one launch per slice of 512 on the stream; every row against the
    oracle, no device flag raised, rows past the last sequence untouched."""
    rng = np.random.default_rng(n_seqs + d)
    lens = [int(n) for n in rng.integers(0, 49, n_seqs)]
    x = W.make_prefill_varlen(lens, 4, 2, d, seed=n_seqs, extra_rows=3)
    kw = {k: v for k, v in variant.items() if k != "alibi"}
    okw = dict(kw)
    if variant.get("alibi"):
        sl = _slopes(4)
        kw["alibi_slopes"] = sl.to(dev)
        okw["alibi_slopes"] = sl.tolist()
    n_q, T, dd = x.q.shape
    o, lse = nan_like((n_q, T, dd), dev), nan_like((n_q, T), dev)
    attn.prefill_varlen(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev), x.scale,
                        True, out=o, lse=lse, **kw)
    attn.check_device_status()
    o_ref, lse_ref = oracle.prefill_varlen(x.q, x.k, x.v, x.cu_seqlens, x.scale, True, **okw)
    T0 = int(x.cu_seqlens[-1])
    compare(o[:, :T0], lse[:, :T0], o_ref[:, :T0], lse_ref[:, :T0], f"{n_seqs} sequences {variant}")
    assert torch.isnan(o[:, T0:]).all() and torch.isnan(lse[:, T0:]).all()


@pytest.mark.parametrize("lens,d,variant", [([1, 127, 0, 129, 300, 45], 128, {}),
                                            ([700, 33, 64], 64, {"window_left": 50}),
                                            ([400, 129, 1], 256, {})])
def test_varlen_bf16_output_is_the_rounded_fp32_output(dev, lens, d, variant):
    """attn_prefill_varlen_ex2 with bf16 O: the rounded fp32 O of the same
    call, bit for bit, including the last boxes of sequences that are written
    row by row; rows outside every sequence untouched."""
    x = W.make_prefill_varlen(lens, 4, 2, d, seed=sum(lens) + d, extra_rows=5)
    q, k, v, cu = x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev)
    n_q, T, _ = x.q.shape
    o32, l32 = attn.prefill_varlen(q, k, v, cu, x.scale, True, **variant)
    o16 = torch.full((n_q, T, d), float("nan"), dtype=torch.bfloat16, device=dev)
    l16 = torch.full((n_q, T), float("nan"), device=dev)
    attn.prefill_varlen(q, k, v, cu, x.scale, True, out=o16, lse=l16, out_dtype=torch.bfloat16,
                        **variant)
    attn.check_device_status()
    T0 = int(x.cu_seqlens[-1])
    assert torch.equal(o16[:, :T0], o32[:, :T0].to(torch.bfloat16))
    assert torch.equal(l16[:, :T0], l32[:, :T0])
    assert torch.isnan(o16[:, T0:].float()).all()
