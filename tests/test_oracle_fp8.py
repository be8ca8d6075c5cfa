"""Pins of the FP8 oracle (oracle/fp8_ref.py): the e4m3 rounding against the
format's definition and torch's conversion, the incoherent rotation against
scipy's Hadamard matrix, the block quantiser's error bound, exactness on
representable inputs, and the method's purpose (lower error than naive
per-tensor FP8 on inputs with outlier channels; page "FlashAttention for
inference", sections "The line of work" and "Interaction with post-trained
models")."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref as F
from exact_io_aware_order_gb300 import workloads as W


def test_round_e4m3_matches_torch_conversion():
    rng = np.random.default_rng(0)
    mags = np.ldexp(1.0, rng.integers(-14, 10, 20000)) * rng.uniform(1, 2, 20000)
    x = (mags * rng.choice([-1, 1], 20000)).astype(np.float32)
    # exact ties and binade edges
    ties = [np.ldexp(1 + (2 * m + 1) / 16, e) for e in range(-6, 8) for m in range(8)]
    x = np.concatenate([x, np.float32(ties), np.float32([0, 448, 449, 464, 480, 1e6, 2 ** -9,
                                                          2 ** -10, 3 * 2 ** -11, 2 ** -6])])
    ours = F.round_e4m3(x)
    theirs = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # torch's conversion turns |x| > 464 (past the midpoint to the next
    # would-be value, 480) into NaN; the GPU's satfinite
    # conversion (and this reference) saturate to +-448 there
    finite = np.abs(x) <= 464
    assert np.array_equal(ours[finite], theirs[finite])
    assert np.all(np.abs(ours[~finite]) == 448.0) and (~finite).sum() > 100


def test_round_e4m3_worked_values():
    cases = {2.0 ** -10: 0.0, 2.0 ** -9: 2.0 ** -9, 1.0625: 1.0, 1.1875: 1.25, 232.0: 224.0,
             248.0: 256.0, 449.0: 448.0, -3.3: -3.25, 0.3: 0.3125, 2.0 ** -6 * 1.0625: 2.0 ** -6}
    for x, want in cases.items():
        assert F.round_e4m3(np.float32(x)) == want, x


def test_hadamard_rotation():
    from scipy.linalg import hadamard

    d = 128
    signs = np.where(np.random.default_rng(1).random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    R = F.hadamard_rotate(np.eye(d, dtype=np.float32), signs).astype(np.float64)
    want = np.diag(signs.astype(np.float64)) @ hadamard(d) / math.sqrt(d)
    assert np.abs(R - want).max() <= 1e-7
    assert np.abs(R @ R.T - np.eye(d)).max() <= 1e-6
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, d)).astype(np.float32)
    k = rng.standard_normal((7, d)).astype(np.float32)
    s0 = q.astype(np.float64) @ k.T.astype(np.float64)
    s1 = F.hadamard_rotate(q, signs).astype(np.float64) @ F.hadamard_rotate(k, signs).T.astype(np.float64)
    assert np.abs(s1 - s0).max() <= 1e-4 * np.abs(s0).max()


def test_quantize_blocks_bound_and_edges():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2, 300, 16)) * np.exp(rng.standard_normal((2, 300, 1)))).astype(np.float32)
    x[1, 128:256] = 0.0                                          # an all-zero block
    codes, scales = F.quantize_blocks(x, 128)
    deq = F.dequantize(codes, scales, 128)
    sc = np.repeat(scales.astype(np.float64), 128, axis=1)[:, :300, None]
    assert np.all(np.abs(deq - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * sc + 1e-12)
    for p in range(2):
        for b in range(3):
            blk = codes[p, b * 128:(b + 1) * 128]
            if np.abs(x[p, b * 128:(b + 1) * 128]).max() > 0:
                assert np.abs(blk).max() == 448.0                  # amax maps to the top code
    assert np.all(codes[1, 128:256] == 0) and scales[1, 1] == np.float32(1.0) / np.float32(448.0)


def test_representable_inputs_pass_through_exactly():
    """Inputs that are e4m3 values with amax 448 in every block quantise to
    themselves with scale 1, so the FP8 reference equals plain attention."""
    rng = np.random.default_rng(4)
    B, nq, nkv, N, d = 1, 2, 1, 256, 16
    def rep(shape):
        x = F.round_e4m3(rng.standard_normal(shape).astype(np.float32) * 40)
        x.reshape(-1, 128 * d if shape[2] >= 128 else shape[2] * d)[:, 0] = 448.0
        return x
    q, k = rep((B, nq, N, d)), rep((B, nkv, N, d))
    v = F.round_e4m3(rng.standard_normal((B, nkv, N, d)).astype(np.float32) * 40)
    v[..., 0, 0] = 448.0
    qz = F.quantize_for_attention(q, k, v)
    assert np.array_equal(qz["qc"], q) and np.all(qz["qs"] == 1.0)
    o8, l8 = F.prefill_fp8(qz, 0.01, True)
    o, l = oracle.prefill(q, k, v, 0.01, True)
    assert np.abs(o8 - o).max() <= 1e-12 and np.abs(l8 - l).max() <= 1e-12


def test_block_and_rotation_lower_the_error():
    """On keys and queries with a few large channels (the outliers the
    rotation spreads), the scores from block-quantised rotated inputs are
    much closer to the exact scores than from naive per-tensor FP8."""
    x = W.make_prefill(1, 4, 2, 512, 128, seed=6)
    q = x.q.double().numpy()
    k = x.k.double().numpy()
    q[..., :4] *= 20.0                                            # outlier channels
    k[..., :4] *= 20.0
    signs = np.where(np.random.default_rng(7).random(128) < 0.5, -1.0, 1.0)
    exact = np.einsum("bhnd,bhmd->bhnm", q[:, :2], k[:, :1].repeat(2, 1))
    def score_err(qz, block):
        qd = F.dequantize(qz["qc"], qz["qs"], block)[:, :2]
        kd = F.dequantize(qz["kc"], qz["ks"], block)[:, :1].repeat(2, 1)
        s = np.einsum("bhnd,bhmd->bhnm", qd, kd)
        return np.sqrt(np.mean((s - exact) ** 2))
    naive = score_err(F.quantize_for_attention(q, k, x.v, None, block=512), 512)
    ours = score_err(F.quantize_for_attention(q, k, x.v, signs, block=128), 128)
    assert naive / ours > 1.5, (naive, ours)


def test_packed_quantisation_matches_each_sequence_alone():
    """Packed FP8 inputs: each sequence's codes and scales equal those of the
    sequence quantised on its own (tiles aligned to its first row), its scales
    sit at the tile prefix of the earlier sequences, rows outside every
    sequence stay 0, and V's per-head scale covers all rows."""
    lens = [130, 0, 16, 257, 5]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1]) + 7
    g = torch.Generator().manual_seed(31)
    q = torch.randn(4, T, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(2, T, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(2, T, 64, generator=g).to(torch.bfloat16)
    signs = np.where(np.random.default_rng(3).random(64) < 0.5, -1.0, 1.0).astype(np.float32)
    qz = F.quantize_for_attention_varlen(q, k, v, cu, signs)
    prefix = F.packed_tile_count(cu)
    assert prefix == [0, 2, 2, 3, 6, 7]
    assert qz["qs"].shape == (4, -(-T // 128) + len(lens))
    for s_, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if b == a:
            continue
        alone = F.quantize_for_attention(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], signs)
        nt = prefix[s_ + 1] - prefix[s_]
        assert np.array_equal(qz["qc"][:, a:b], alone["qc"][0])
        assert np.array_equal(qz["kc"][:, a:b], alone["kc"][0])
        assert np.array_equal(qz["qs"][:, prefix[s_]:prefix[s_] + nt], alone["qs"][0])
        assert np.array_equal(qz["ks"][:, prefix[s_]:prefix[s_] + nt], alone["ks"][0])
    assert not qz["qc"][:, int(cu[-1]):].any() and not qz["qs"][:, prefix[-1]:].any()
    whole = F.quantize_for_attention(q[None], k[None], v[None])
    assert np.array_equal(qz["vc"], whole["vc"][0]) and np.array_equal(qz["vs"], whole["vs"][0])


def test_packed_fp8_attention_equals_per_sequence_fp8_attention():
    """The packed FP8 attention is, sequence by sequence, the FP8 attention of
    the sequence alone with V's scale of the whole packed tensor."""
    lens = [40, 0, 97]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, T, 16, generator=g).to(torch.bfloat16)
    k = torch.randn(1, T, 16, generator=g).to(torch.bfloat16)
    v = torch.randn(1, T, 16, generator=g).to(torch.bfloat16)
    qz = F.quantize_for_attention_varlen(q, k, v, cu)
    for causal in (True, False):
        o, lse = F.prefill_fp8_varlen(qz, 0.25, causal)
        for a, b in zip(cu[:-1], cu[1:]):
            if b == a:
                continue
            alone = F.quantize_for_attention(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b])
            alone["vc"] = qz["vc"][None, :, a:b]
            alone["vs"] = qz["vs"][None]
            oa, la = F.prefill_fp8(alone, 0.25, causal)
            assert np.abs(oa[0] - o[:, a:b]).max() <= 1e-12
            assert np.abs(la[0] - lse[:, a:b]).max() <= 1e-12
