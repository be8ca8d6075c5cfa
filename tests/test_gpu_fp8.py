"""FP8 path on the GPU against the float64 / exact-float32 oracle
(oracle/fp8_ref.py): the quantiser's e4m3 codes and scales bit for bit
(rotated or not, per block or per plane, row-major or transposed)."""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from oracle import fp8_ref as F

pytestmark = pytest.mark.gpu


def e4m3_values(codes_u8):
    return codes_u8.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def signs_for(d, seed):
    return np.where(np.random.default_rng(seed).random(d) < 0.5, -1.0, 1.0).astype(np.float32)


@pytest.mark.parametrize("planes,rows,d,rot,block,transpose", [
    (3, 300, 128, True, 128, False),
    (2, 256, 128, False, 128, True),
    (4, 1000, 128, False, 0, True),
    (2, 129, 64, True, 128, False),
    (1, 4096, 128, True, 0, False),
    (3, 4100, 64, True, 0, True),      # per-plane scale, transposed, rows not a multiple of 16
    (2, 8192, 128, True, 0, True),
    (5, 17, 128, True, 128, True),     # one partial block
    (40, 2000, 128, True, 128, False),  # more blocks than CTAs (staged, several per CTA), ragged ends
    (48, 1100, 64, False, 128, False),  # the same at head_dim 64
    (24, 3000, 64, True, 0, True),      # per-plane amax over many staged blocks
])
def test_quantizer_bit_exact(dev, planes, rows, d, rot, block, transpose):
    g = torch.Generator().manual_seed(rows + d)
    x = (torch.randn(planes, rows, d, generator=g) *
         torch.exp(torch.randn(planes, rows, 1, generator=g))).to(torch.bfloat16)
    x[0, :, 3] *= 30                                           # an outlier channel
    sg = signs_for(d, 5) if rot else None
    codes, scales = attn.quantize_fp8(x.to(dev), torch.from_numpy(sg).to(dev) if rot else None,
                                      block_rows=block, transpose=transpose)
    attn.check_device_status()
    x32 = x.float().numpy()
    if rot:
        x32 = F.hadamard_rotate(x32, sg)
    ref_codes, ref_scales = F.quantize_blocks(x32, block if block else rows)
    got = e4m3_values(codes)
    if transpose:
        got = got.transpose(0, 2, 1)
    assert np.array_equal(got, ref_codes)
    assert np.array_equal(scales.cpu().numpy().reshape(ref_scales.shape), ref_scales)


@pytest.mark.parametrize("pq,pk,rows,d,rot", [
    (28, 4, 8192, 128, True),     # the Qwen2.5-7B layer's Q, K and V at N = 8192
    (3, 1, 300, 64, False),
    (6, 3, 4100, 128, True),      # rows not a multiple of 16
    (2, 2, 17, 128, True),        # one partial block
])
def test_quantizer_qkv_matches_separate_calls_and_oracle(dev, pq, pk, rows, d, rot):
    """attn_quantize_fp8_qkv: bit for bit the three attn_quantize_fp8 calls
    (Q, K block-scaled and rotated, V per plane and transposed), and the
    oracle's codes and scales."""
    g = torch.Generator().manual_seed(pq + rows)
    mk = lambda p: (torch.randn(p, rows, d, generator=g) *
                    torch.exp(torch.randn(p, rows, 1, generator=g))).to(torch.bfloat16)
    q, k, v = mk(pq), mk(pk), mk(pk)
    k[0, :, 5] *= 25                                           # an outlier channel
    sg = signs_for(d, 7) if rot else None
    sgd = torch.from_numpy(sg).to(dev) if rot else None
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fused = attn.quantize_fp8_qkv(qd, kd, vd, sgd)
    sep = (*attn.quantize_fp8(qd, sgd, block_rows=128)[:1], *attn.quantize_fp8(kd, sgd, 128)[:1],
           *attn.quantize_fp8(vd, None, 0, True)[:1])
    sep_s = (attn.quantize_fp8(qd, sgd, 128)[1], attn.quantize_fp8(kd, sgd, 128)[1],
             attn.quantize_fp8(vd, None, 0, True)[1])
    attn.check_device_status()
    for a, b in zip(fused[:3], sep):
        assert torch.equal(a, b)
    for a, b in zip(fused[3:], sep_s):
        assert torch.equal(a, b)
    # against the oracle
    for x, codes, scales, block, tr, rot_ in ((q, fused[0], fused[3], 128, False, rot),
                                              (k, fused[1], fused[4], 128, False, rot),
                                              (v, fused[2], fused[5], rows, True, False)):
        x32 = x.float().numpy()
        if rot_:
            x32 = F.hadamard_rotate(x32, sg)
        ref_codes, ref_scales = F.quantize_blocks(x32, block)
        got = e4m3_values(codes)
        if tr:
            got = got.transpose(0, 2, 1)
        assert np.array_equal(got, ref_codes)
        assert np.array_equal(scales.cpu().numpy().reshape(ref_scales.shape), ref_scales)


@pytest.mark.parametrize("block", [128, 0])
def test_quantizer_all_zero_plane(dev, block):
    """A block (or plane) of zeros: amax 0 counts as 1, so its scale is 1/448
    and its codes are 0."""
    x = torch.zeros(3, 200, 128, dtype=torch.bfloat16)
    x[1] = torch.randn(200, 128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    codes, scales = attn.quantize_fp8(x.to(dev), None, block_rows=block)
    attn.check_device_status()
    ref_codes, ref_scales = F.quantize_blocks(x.float().numpy(), block if block else 200)
    assert np.array_equal(e4m3_values(codes), ref_codes)
    assert np.array_equal(scales.cpu().numpy().reshape(ref_scales.shape), ref_scales)
    assert np.all(scales.cpu().numpy()[0] == np.float32(1.0) / np.float32(448.0))


def fp8_inputs(x, dev, signs, block=128):
    """GPU FP8 inputs of a prefill workload: rotated + block-quantised Q, K,
    per-head V (transposed)."""
    sg = torch.from_numpy(signs).to(dev) if signs is not None else None
    q8, qs = attn.quantize_fp8(x.q.to(dev), sg, block_rows=block)
    k8, ks = attn.quantize_fp8(x.k.to(dev), sg, block_rows=block)
    v8t, vs = attn.quantize_fp8(x.v.to(dev), None, block_rows=0, transpose=True)
    if block == 0:   # one scale per head for Q and K too: present it per block
        nb = -(-x.q.shape[2] // 128)
        qs = qs.unsqueeze(-1).expand(*qs.shape, nb).contiguous()
        ks = ks.unsqueeze(-1).expand(*ks.shape, nb).contiguous()
    return q8, k8, v8t, qs, ks, vs


def p_rounding_sigma(qz, scale, causal):
    """Predicted rms of the O error from rounding P to e4m3: each P is off by
    a relative error uniform in +-2^-4 (rms 2^-4 / sqrt 3), so
    sigma_ij = 0.036 sqrt(sum_k P_ik^2 v_kj^2) with P normalised."""
    qd = F.dequantize(qz["qc"], qz["qs"], 128)
    kd = F.dequantize(qz["kc"], qz["ks"], 128)
    vd = qz["vc"] * np.asarray(qz["vs"], dtype=np.float64)[..., None, None]
    B, nq, N, d = qd.shape
    g = nq // kd.shape[1]
    sig = np.zeros(qd.shape)
    for b in range(B):
        for h in range(nq):
            s = scale * qd[b, h] @ kd[b, h // g].T
            if causal:
                s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            sig[b, h] = (2.0 ** -4 / np.sqrt(3.0)) * np.sqrt((p ** 2) @ (vd[b, h // g] ** 2))
    return sig


@pytest.mark.parametrize("B,N,Hq,Hkv,causal,d", [(1, 1024, 8, 2, True, 128),
                                                 (1, 768, 4, 4, False, 128),
                                                 (1, 2048, 4, 1, True, 128),
                                                 (2, 640, 6, 2, True, 128),   # a batch: scales per
                                                 (3, 400, 4, 1, False, 64),   # (sequence, head, tile)
                                                 (1, 1024, 8, 2, True, 64),   # 64 columns: the
                                                 (1, 640, 4, 4, False, 64),   # 128-wide tiles read
                                                 (1, 336, 6, 3, True, 64)])   # zeros past them
def test_prefill_fp8_parity(dev, B, N, Hq, Hkv, causal, d):
    from exact_io_aware_order_gb300 import workloads as W

    x = W.make_prefill(B, Hq, Hkv, N, d, seed=N + Hq + B, causal=causal)
    signs = signs_for(d, 11)
    q8, k8, v8t, qs, ks, vs = fp8_inputs(x, dev, signs)
    o, lse = attn.prefill_fp8(q8, k8, v8t, qs, ks, vs, x.scale, causal)
    attn.check_device_status()
    qz = F.quantize_for_attention(x.q, x.k, x.v, signs)
    # the GPU's codes are the oracle's (checked bit for bit above); the attention:
    o_ref, lse_ref = F.prefill_fp8(qz, x.scale, causal)
    lerr = np.abs(lse.double().cpu().numpy() - lse_ref).max()
    assert lerr <= 1e-3, lerr
    sig = p_rounding_sigma(qz, x.scale, causal)
    err = np.abs(o.double().cpu().numpy() - o_ref)
    z = err / (sig + 1e-6)
    assert z.max() <= 6.0, (z.max(), err.max())
    assert z.mean() <= 1.0, z.mean()                 # ~0.8 for normally distributed errors


def test_fp8_block_quantisation_and_rotation_lower_the_error(dev):
    """Against exact attention on the unquantised inputs, the GPU FP8 path
    with block scales and the rotation errs much less than with one scale per
    head and no rotation, on queries and keys with outlier channels."""
    from exact_io_aware_order_gb300 import workloads as W
    import oracle

    x = W.make_prefill(1, 8, 2, 1024, 128, seed=3)
    x.q[..., :4] *= 20.0
    x.k[..., :4] *= 20.0
    o_exact, _ = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    errs = {}
    for name, signs, block in (("naive", None, 0), ("block+rotation", signs_for(128, 2), 128)):
        o, _ = attn.prefill_fp8(*fp8_inputs(x, dev, signs, block), x.scale, True)
        errs[name] = np.sqrt(np.mean((o.double().cpu().numpy() - o_exact) ** 2))
    attn.check_device_status()
    assert errs["naive"] / errs["block+rotation"] > 1.5, errs


def test_packed_quantizer_bit_exact(dev):
    """attn_quantize_fp8_varlen: codes and scales of packed rows equal the
    oracle's bit for bit (tiles from each sequence's first row; scale columns
    at the tile prefix); rows outside every sequence and unused columns stay
    zero."""
    lens = [130, 0, 16, 257, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1]) + 9
    g = torch.Generator().manual_seed(12)
    for d, rot in ((128, True), (64, False)):
        x = torch.randn(3, T, d, generator=g).to(torch.bfloat16)
        signs = signs_for(d, 4) if rot else None
        sg = torch.from_numpy(signs).to(dev) if rot else None
        codes, scales = attn.quantize_fp8_varlen(x.to(dev), torch.from_numpy(cu).to(dev), sg)
        attn.check_device_status()
        ref = F.quantize_for_attention_varlen(x, x[:1], x[:1], cu, signs)
        assert np.array_equal(e4m3_values(codes), ref["qc"])
        assert np.array_equal(scales.cpu().numpy(), ref["qs"])


def packed_sigma(qz, scale, causal):
    """p_rounding_sigma sequence by sequence (each with its own tiles' scales)."""
    prefix = F.packed_tile_count(qz["cu"])
    sig = np.zeros(qz["qc"].shape)
    for s_, (a, b) in enumerate(zip(qz["cu"][:-1], qz["cu"][1:])):
        if b == a:
            continue
        nt = prefix[s_ + 1] - prefix[s_]
        one = {"qc": qz["qc"][None, :, a:b], "qs": qz["qs"][None, :, prefix[s_]:prefix[s_] + nt],
               "kc": qz["kc"][None, :, a:b], "ks": qz["ks"][None, :, prefix[s_]:prefix[s_] + nt],
               "vc": qz["vc"][None, :, a:b], "vs": qz["vs"][None]}
        sig[:, a:b] = p_rounding_sigma(one, scale, causal)[0]
    return sig


@pytest.mark.parametrize("lens,Hq,Hkv,causal,d", [([256, 0, 48, 144, 37], 8, 2, True, 128),
                                                  ([512, 16, 160], 4, 4, False, 128),
                                                  ([32, 1000], 4, 1, True, 128),
                                                  ([256, 0, 48, 144, 37], 8, 2, True, 64),
                                                  ([512, 16, 160], 4, 4, False, 64)])
def test_prefill_fp8_varlen_parity(dev, lens, Hq, Hkv, causal, d):
    """Packed FP8 prefill (every sequence starting at a multiple of 16 rows)
    against the oracle's packed FP8 attention: LSE within 1e-3, O within the
    P-rounding bound, rows past the last sequence untouched."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = -(-int(cu[-1]) // 16) * 16 + 16
    g = torch.Generator().manual_seed(sum(lens) + Hq)
    q = torch.randn(Hq, T, d, generator=g).to(torch.bfloat16)
    k = torch.randn(Hkv, T, d, generator=g).to(torch.bfloat16)
    v = torch.randn(Hkv, T, d, generator=g).to(torch.bfloat16)
    signs = signs_for(d, 21)
    sg = torch.from_numpy(signs).to(dev)
    cud = torch.from_numpy(cu).to(dev)
    q8, qs = attn.quantize_fp8_varlen(q.to(dev), cud, sg)
    k8, ks = attn.quantize_fp8_varlen(k.to(dev), cud, sg)
    v8t, vs = attn.quantize_fp8(v.to(dev), None, block_rows=0, transpose=True)
    scale = 1.0 / math.sqrt(d)
    o = torch.full((Hq, T, d), float("nan"), device=dev)
    lse = torch.full((Hq, T), float("nan"), device=dev)
    attn.prefill_fp8_varlen(q8, k8, v8t, qs, ks, vs, cud, scale, causal, out=o, lse=lse)
    attn.check_device_status()
    qz = F.quantize_for_attention_varlen(q, k, v, cu, signs)
    o_ref, lse_ref = F.prefill_fp8_varlen(qz, scale, causal)
    T0 = int(cu[-1])
    lerr = np.abs(lse[:, :T0].double().cpu().numpy() - lse_ref[:, :T0]).max()
    assert lerr <= 1e-3, lerr
    sig = packed_sigma(qz, scale, causal)[:, :T0]
    z = np.abs(o[:, :T0].double().cpu().numpy() - o_ref[:, :T0]) / (sig + 1e-6)
    assert z.max() <= 6.0 and z.mean() <= 1.0, (z.max(), z.mean())
    assert torch.isnan(o[:, T0:]).all() and torch.isnan(lse[:, T0:]).all()


def test_prefill_fp8_varlen_misaligned_start_is_refused(dev):
    """A non-empty sequence that starts off a multiple of 16 rows: the kernel
    checks cu_seqlens before any copy, computes nothing and flags the launch."""
    T, d = 64, 128
    cu = torch.tensor([0, 20, 64], dtype=torch.int32, device=dev)   # second sequence at row 20
    z8 = torch.zeros((2, T, d), dtype=torch.uint8, device=dev)
    v8t = torch.zeros((2, d, T), dtype=torch.uint8, device=dev)
    sc = torch.ones((2, 3), dtype=torch.float32, device=dev)
    vs = torch.ones(2, dtype=torch.float32, device=dev)
    o = torch.full((2, T, d), float("nan"), device=dev)
    lse = torch.full((2, T), float("nan"), device=dev)
    attn.prefill_fp8_varlen(z8, z8, v8t, sc, sc, vs, cu, 0.1, True, out=o, lse=lse)
    with pytest.raises(attn.AttnError):
        attn.check_device_status()
    assert torch.isnan(o).all() and torch.isnan(lse).all()


def test_prefill_fp8_qwen_8192_sampled(dev):
    """The benchmarked FP8 shape (Qwen2.5-7B layer, N = 8192, 28 / 4 heads,
    block scales + rotation): 300 sampled rows against exact attention on the
    dequantised inputs; LSE within 1e-3, O within the P-rounding bound of
    those rows."""
    from exact_io_aware_order_gb300 import workloads as W
    import oracle

    x = W.qwen_prefill(8192)
    signs = signs_for(128, 11)
    q8, k8, v8t, qs, ks, vs = fp8_inputs(x, dev, signs)
    o, lse = attn.prefill_fp8(q8, k8, v8t, qs, ks, vs, x.scale, True)
    attn.check_device_status()
    qz = F.quantize_for_attention(x.q, x.k, x.v, signs)
    qd = F.dequantize(qz["qc"], qz["qs"], 128)
    kd = F.dequantize(qz["kc"], qz["ks"], 128)
    vd = qz["vc"] * np.asarray(qz["vs"], dtype=np.float64)[..., None, None]
    rng = np.random.default_rng(8)
    rows = [(0, int(h), int(i)) for h, i in zip(rng.integers(0, 28, 300), rng.integers(0, 8192, 300))]
    o_ref, lse_ref = oracle.prefill_rows(qd, kd, vd, x.scale, True, rows)
    idx = tuple(torch.tensor(c) for c in zip(*rows))
    lerr = np.abs(lse[idx].double().cpu().numpy() - lse_ref).max()
    assert lerr <= 1e-3, lerr
    sig = np.zeros(o_ref.shape)
    for r, (b, h, i) in enumerate(rows):
        kh = h // 7
        s = x.scale * (kd[b, kh, :i + 1] @ qd[b, h, i])
        p = np.exp(s - s.max())
        p /= p.sum()
        sig[r] = (2.0 ** -4 / np.sqrt(3.0)) * np.sqrt((p ** 2) @ (vd[b, kh, :i + 1] ** 2))
    z = np.abs(o[idx].double().cpu().numpy() - o_ref) / (sig + 1e-6)
    assert z.max() <= 6.0 and z.mean() <= 1.0, (z.max(), z.mean())
