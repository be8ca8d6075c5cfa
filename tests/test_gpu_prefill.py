"""Parity of the sm_103a prefill kernel (attn_prefill, through the C ABI)
against the float64 oracle: every element at small and ragged sizes, every
row of some heads plus random rows of all heads at the full workload sizes."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
import oracle
from gpu_util import compare, nan_like

pytestmark = pytest.mark.gpu


def run_prefill(x, dev, causal=None):
    causal = x.causal if causal is None else causal
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    B, Hq, N, D = q.shape
    o = nan_like((B, Hq, N, D), dev)      # unwritten elements would stay NaN
    lse = nan_like((B, Hq, N), dev)
    attn.prefill(q, k, v, x.scale, causal, out=o, lse=lse)
    attn.check_device_status()
    return o, lse


def test_tiny_causal_prefill(dev):
    """Batch 1, 1 head, N=256, head_dim 64."""
    x = W.tiny_prefill()
    o, lse = run_prefill(x, dev)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    compare(o, lse, o_ref, lse_ref, "tiny")


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal", [
    (1, 1, 1, 1, 64, True), (1, 1, 1, 7, 128, True), (1, 2, 1, 100, 128, True),
    (1, 1, 1, 128, 64, True), (1, 1, 1, 129, 128, True), (2, 4, 2, 300, 128, True),
    (1, 3, 3, 383, 64, True), (1, 2, 2, 511, 128, True), (1, 2, 1, 1000, 128, True),
    (1, 7, 1, 640, 128, True), (1, 2, 1, 700, 128, False), (2, 2, 2, 256, 64, False),
    (1, 1, 1, 5, 128, False), (3, 2, 1, 257, 64, True),
    (16, 32, 8, 200, 128, True)])              # 512 planes: several items per CTA
def test_ragged_and_small_shapes(dev, B, Hq, Hkv, N, D, causal):
    x = W.make_prefill(B, Hq, Hkv, N, D, seed=N + 7 * D + B)
    o, lse = run_prefill(x, dev, causal)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal)
    compare(o, lse, o_ref, lse_ref, f"B{B} H{Hq}/{Hkv} N{N} D{D} causal{causal}")


def test_qwen_2048_every_element(dev):
    """Qwen2.5-7B layer shape (28 / 4 heads, head_dim 128), N=2048."""
    x = W.qwen_prefill(2048)
    o, lse = run_prefill(x, dev)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    compare(o, lse, o_ref, lse_ref, "qwen 2048")


def _sampled(x, o, lse, heads_full, rows_per_head, seed):
    B, Hq, N, D = x.q.shape
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        for h in range(Hq):
            if h in heads_full:
                idx = range(N)
            else:
                idx = sorted(set(rng.integers(0, N, rows_per_head).tolist()) | {0, N - 1, min(N - 1, 128), min(N - 1, 255)})
            rows += [(b, h, int(i)) for i in idx]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, x.causal, rows)
    bi = torch.tensor([r[0] for r in rows]); hi = torch.tensor([r[1] for r in rows])
    ii = torch.tensor([r[2] for r in rows])
    og = o.cpu()[bi, hi, ii]
    lg = lse.cpu()[bi, hi, ii]
    return compare(og, lg, o_ref, lse_ref, "sampled")


def test_qwen_8192_sampled_rows(dev):
    """N=8192: every row of two heads, 256 random rows (plus edges) of the rest."""
    x = W.qwen_prefill(8192)
    o, lse = run_prefill(x, dev)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    _sampled(x, o, lse, heads_full={0, 27}, rows_per_head=256, seed=1)


@pytest.mark.parametrize("N", [30720, 32768])
def test_llama_long_spiky_sampled_rows(dev, N):
    """Llama-3-8B layer (32 / 8 heads) at long context, 1% of keys scaled by 8."""
    x = W.llama_long_prefill(N)
    o, lse = run_prefill(x, dev)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    _sampled(x, o, lse, heads_full=set(), rows_per_head=48, seed=N)


def test_long_sequence_131072_sampled(dev):
    """N = 131072 (1024 query tiles per plane, row indices past 2^16, a
    causal row reading up to 1024 key tiles), 1% of the keys x8: sampled rows,
    among them the first and last rows and the tile and 2^16 boundaries,
    against the oracle."""
    N = 131072
    x = W.make_prefill(1, 2, 1, N, 128, seed=13, spike_frac=0.01)
    o, lse = run_prefill(x, dev)
    rows = [(0, h, i) for h in (0, 1) for i in (0, 1, 127, 128, 65535, 65536, N - 2, N - 1)]
    rng = np.random.default_rng(13)
    rows += [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 2, 100), rng.integers(0, N, 100))]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, True, rows)
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    compare(o[idx], lse[idx], o_ref, lse_ref, "N=131072 spiky")


def test_batch_with_l2_grouping_sampled(dev):
    """Batch 2 of Llama-3-8B layers at N = 16384 (32 / 8 heads): K and V take
    134 MB, so the work list runs in groups of two kv heads (8 query planes)
    for L2 locality, eight groups over the batch; sampled rows of both
    sequences against the oracle."""
    x = W.make_prefill(2, 32, 8, 16384, 128, seed=17, spike_frac=0.01)
    o, lse = run_prefill(x, dev)
    rng = np.random.default_rng(17)
    rows = [(int(b), int(h), int(i)) for b, h, i in
            zip(rng.integers(0, 2, 160), rng.integers(0, 32, 160), rng.integers(0, 16384, 160))]
    rows += [(1, 31, 16383), (1, 0, 0), (0, 31, 16383)]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, True, rows)
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    compare(o[idx], lse[idx], o_ref, lse_ref, "B=2 N=16384 grouped")


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,variant", [
    (1, 4, 2, 1000, 128, True, {}),
    (2, 2, 1, 300, 64, False, {}),
    (1, 2, 2, 700, 256, True, {}),
    (1, 4, 1, 900, 128, True, {"window_left": 200}),
    (1, 4, 2, 600, 128, True, {"softcap": 30.0}),
    (1, 4, 2, 640, 128, False, {"alibi": True}),
])
def test_bf16_output_is_the_rounded_fp32_output(dev, B, Hq, Hkv, N, D, causal, variant):
    """attn_prefill_ex2 with ATTN_PREFILL_OUT_BF16: O is acc / l rounded once
    to bf16, so it equals the fp32 O of the same inputs rounded to nearest,
    bit for bit, and the LSE is unchanged."""
    x = W.make_prefill(B, Hq, Hkv, N, D, seed=N + D + B, causal=causal)
    kw = {k_: v_ for k_, v_ in variant.items() if k_ != "alibi"}
    if variant.get("alibi"):
        kw["alibi_slopes"] = torch.tensor([2.0 ** (-(h + 1)) for h in range(Hq)],
                                          dtype=torch.float32, device=dev)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o32, l32 = attn.prefill(q, k, v, x.scale, causal, **kw)
    o16 = torch.full((B, Hq, N, D), float("nan"), dtype=torch.bfloat16, device=dev)
    o16, l16 = attn.prefill(q, k, v, x.scale, causal, out=o16, out_dtype=torch.bfloat16, **kw)
    attn.check_device_status()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)


def test_closed_forms_on_gpu(dev):
    """q = 0 gives LSE_i = ln(i+1) and O_i = mean(v_0..v_i); V = 1 gives O = 1."""
    x = W.make_prefill(1, 2, 1, 700, 128, seed=3)
    x.q.zero_()
    o, lse = run_prefill(x, dev)
    N = 700
    v = x.v[0, 0].double().numpy()
    pm = np.cumsum(v, 0) / np.arange(1, N + 1)[:, None]
    ref_l = np.log(np.arange(1, N + 1))
    compare(o[0], lse[0], np.stack([pm, pm]), np.stack([ref_l, ref_l]), "q=0")
    # V = 1: O = 1 up to the rounding of P to bf16 before the P V product
    # (l is summed from the unrounded P), i.e. within the usual tolerance.
    y = W.make_prefill(1, 2, 2, 333, 64, seed=4)
    y.v.fill_(1.0)
    o1, l1 = run_prefill(y, dev)
    o_ref, l_ref = oracle.prefill(y.q, y.k, y.v, y.scale, True)
    assert np.abs(o_ref - 1.0).max() <= 1e-13
    compare(o1, l1, o_ref, l_ref, "V=1")


def test_repeated_launch_is_deterministic(dev):
    x = W.make_prefill(1, 4, 2, 1500, 128, seed=5)
    o1, l1 = run_prefill(x, dev)
    o2, l2 = run_prefill(x, dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [
    (1, 4, 1, 1000, True),     # ragged tail, GQA 4:1
    (2, 2, 2, 384, True),      # batch, MHA, whole tiles
    (1, 8, 2, 777, False),     # full attention
    (1, 2, 1, 64, True),       # one 64-key tile
    (1, 16, 2, 2048, True),
])
def test_head_dim_256(dev, B, Hq, Hkv, N, causal):
    """head_dim 256 (one of the variants the page lists): 64-key tiles, O in
    256 TMEM columns, the epilogue in two halves."""
    x = W.make_prefill(B, Hq, Hkv, N, 256, seed=N + Hq, causal=causal)
    o, lse = run_prefill(x, dev)
    o_ref, lse_ref = oracle.prefill(x.q, x.k, x.v, x.scale, causal)
    compare(o, lse, o_ref, lse_ref, f"d=256 B={B} N={N}")


@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_256_8192_spiky_sampled(dev, causal):
    """The benchmarked head_dim-256 shape (N = 8192, 16 / 8 heads) with 1% of
    the keys x8 (the running max jumps, so O is rescaled part-way): 400
    sampled rows against the oracle."""
    x = W.make_prefill(1, 16, 8, 8192, 256, seed=5, spike_frac=0.01, causal=causal)
    o, lse = run_prefill(x, dev, causal)
    rng = np.random.default_rng(9)
    rows = [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 16, 400), rng.integers(0, 8192, 400))]
    o_ref, lse_ref = oracle.prefill_rows(x.q, x.k, x.v, x.scale, causal, rows)
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    compare(o[idx], lse[idx], o_ref, lse_ref, f"d=256 N=8192 spiky causal={causal}")
