"""FP8 (e4m3) block quantisation with incoherent processing, and the
attention it feeds: the float64 / exact-float32 reference.

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` leg are the only callers; the CUDA library never
routes through this file and this file imports nothing from the library.

Source: the explainer page "FlashAttention for inference: tiled prefill and
split-KV decoding" (pofe.ai).  Its section "Interaction with post-trained
models" says that FlashAttention-3's FP8 path reduces the error of naive FP8
attention by block quantisation and incoherent processing, and its section
"The line of work" that this gives 2.6x lower FP8 error than a baseline FP8
attention.  The page names the two techniques without their details, so the
reading taken here (listed with its reasons in the design notes) is:

* incoherent processing: Q and K are multiplied along the head dimension by
  the same orthogonal matrix R = diag(signs) H / sqrt(d), H the Sylvester
  Hadamard matrix and signs a seeded +-1 vector, so Q R (K R)^T = Q K^T while
  outliers are spread over all coordinates;
* block quantisation: Q and K get one scale per 128-row block of each head,
  V one scale per head; a block's scale is amax / 448 (448 = the largest e4m3
  value), its codes are e4m3(x * (448 / amax)), rounded to nearest, ties to
  even, saturating;
* the attention then runs on the dequantised Q R, K R and V with the usual
  scale.  (The GPU path also rounds P to e4m3 for the P V product; the
  reference keeps P exact, and the tests bound the difference.)

Every quantisation step is written with the float32 operations, in the
order, that the GPU quantiser uses, so that both take the same rounding
decisions and the codes can be compared bit for bit.
"""

from __future__ import annotations

import numpy as np

from .attention_ref import _f64, _seq_bounds, prefill, prefill_varlen

__all__ = ["E4M3_MAX", "round_e4m3", "hadamard_rotate", "quantize_blocks",
           "quantize_for_attention", "prefill_fp8", "quantize_for_attention_varlen",
           "prefill_fp8_varlen"]

E4M3_MAX = 448.0
_BLOCK = 128


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3 value of each float32 input (ties to even), saturating at
    +-448.  e4m3: 4 exponent bits (bias 7) and 3 mantissa bits, so normal
    values 2^-6 .. 448 are spaced 2^(e-3) within the binade [2^e, 2^(e+1)),
    and subnormals are the multiples of 2^-9 below 2^-6.  Returns float64
    holding the exact e4m3 values."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))        # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)                       # binade exponent, subnormal floor
    ulp = np.ldexp(1.0, e - 3)
    q = np.round(a / ulp) * ulp                      # a / ulp is exact; np.round is half-even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def hadamard_rotate(x, signs) -> np.ndarray:
    """x (..., d) float32 times diag(signs) H / sqrt(d), in float32: the signs
    first, then the fast Walsh-Hadamard butterflies with stride h = 1, 2, 4,
    ..., d/2 ((a, b) -> (a + b, a - b) for the pair of indices (i, i + h) in
    each block of 2h), then one multiply by the float32 value of 1/sqrt(d)."""
    y = (np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)).astype(np.float32)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("head_dim must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(*lead, d // (2 * h), 2, h)
        a, b = y[..., 0, :], y[..., 1, :]
        y = np.stack((a + b, a - b), axis=-2).reshape(*lead, d)
        h *= 2
    return (y * np.float32(1.0 / np.sqrt(d))).astype(np.float32)


def quantize_blocks(x, block: int):
    """x (planes, rows, d) float32.  Per plane and per block of `block` rows:
    amax = max |x| (1 where the block is all zero), inv = 448 / amax and
    scale = amax / 448 (float32 divisions), codes = e4m3(x * inv) (float32
    multiply).  Returns (codes (planes, rows, d) float64 e4m3 values,
    scales (planes, ceil(rows / block)) float32)."""
    x = np.asarray(x, dtype=np.float32)
    P, R, d = x.shape
    nb = -(-R // block)
    codes = np.zeros(x.shape, dtype=np.float64)
    scales = np.zeros((P, nb), dtype=np.float32)
    for p in range(P):
        for b in range(nb):
            blk = x[p, b * block:(b + 1) * block]
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            if amax == 0:
                amax = np.float32(1.0)
            inv = np.float32(E4M3_MAX) / amax
            scales[p, b] = amax / np.float32(E4M3_MAX)
            codes[p, b * block:(b + 1) * block] = round_e4m3((blk * inv).astype(np.float32))
    return codes, scales


def quantize_for_attention(q, k, v, signs=None, block: int = _BLOCK):
    """The FP8 inputs of the attention: q (B, n_q, N, d), k, v (B, n_kv, N, d)
    (bf16 or float values).  With `signs` (d,) the incoherent rotation is
    applied to q and k first; q and k are quantised per `block` rows of each
    head (block=N: one scale per head, the naive scheme), v per head.
    Returns dict with codes and scales: qc (B, n_q, N, d), qs (B, n_q, nb),
    kc, ks likewise, vc (B, n_kv, N, d), vs (B, n_kv)."""
    q32 = _f64(q).astype(np.float32)
    k32 = _f64(k).astype(np.float32)
    v32 = _f64(v).astype(np.float32)
    if signs is not None:
        q32 = hadamard_rotate(q32, signs)
        k32 = hadamard_rotate(k32, signs)
    B, nq, N, d = q32.shape
    nkv = k32.shape[1]
    qc, qs = quantize_blocks(q32.reshape(B * nq, N, d), block)
    kc, ks = quantize_blocks(k32.reshape(B * nkv, N, d), block)
    vc, vs = quantize_blocks(v32.reshape(B * nkv, N, d), N)
    return {"qc": qc.reshape(B, nq, N, d), "qs": qs.reshape(B, nq, -1),
            "kc": kc.reshape(B, nkv, N, d), "ks": ks.reshape(B, nkv, -1),
            "vc": vc.reshape(B, nkv, N, d), "vs": vs.reshape(B, nkv)}


def dequantize(codes, scales, block: int) -> np.ndarray:
    """codes (..., rows, d) times the scale of each row's block."""
    rows = codes.shape[-2]
    per_row = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=-1)[..., :rows]
    return codes * per_row[..., None]


def prefill_fp8(qz: dict, scale: float, causal: bool = True, block: int = _BLOCK):
    """Attention (the plain definition of :func:`attention_ref.prefill`) on
    the dequantised FP8 inputs of :func:`quantize_for_attention`."""
    N = qz["qc"].shape[2]
    qd = dequantize(qz["qc"], qz["qs"], block)
    kd = dequantize(qz["kc"], qz["ks"], block)
    vd = qz["vc"] * np.asarray(qz["vs"], dtype=np.float64)[..., None, None]
    return prefill(qd, kd, vd, scale, causal)


def packed_tile_count(cu_seqlens, block: int = _BLOCK) -> list:
    """Per packed sequence, the first index of its tiles in the scale arrays
    of :func:`quantize_for_attention_varlen`: sequence s's tile t is column
    prefix[s] + t, prefix[s] = sum over the earlier sequences of
    ceil(len / block).  Returns the prefix list (num_seqs + 1 entries)."""
    prefix = [0]
    for a, b in _seq_bounds(cu_seqlens):
        prefix.append(prefix[-1] + -(-(b - a) // block))
    return prefix


def quantize_for_attention_varlen(q, k, v, cu_seqlens, signs=None, block: int = _BLOCK):
    """The FP8 inputs of a packed prefill: q (n_q, total, d), k, v (n_kv,
    total, d) with sequence s on rows [cu[s], cu[s+1]).  Q and K (rotated
    with `signs` first) are quantised per tile of `block` rows of each
    sequence, tiles starting at the sequence's first row, so that a tile of
    the attention never straddles two scales; the scale of sequence s's tile
    t is column prefix[s] + t (:func:`packed_tile_count`) of an array with
    ceil(total / block) + num_seqs columns (the rest stay 0).  Rows outside
    every sequence are not quantised (codes 0).  V: one scale per head over
    all its rows, as in :func:`quantize_for_attention`.
    Returns dict: qc (n_q, total, d), qs (n_q, width), kc, ks likewise,
    vc (n_kv, total, d), vs (n_kv,)."""
    q32 = _f64(q).astype(np.float32)
    k32 = _f64(k).astype(np.float32)
    v32 = _f64(v).astype(np.float32)
    if signs is not None:
        q32 = hadamard_rotate(q32, signs)
        k32 = hadamard_rotate(k32, signs)
    nq, T, d = q32.shape
    nkv = k32.shape[0]
    bounds = _seq_bounds(cu_seqlens)
    width = -(-T // block) + len(bounds)
    prefix = packed_tile_count(cu_seqlens, block)
    out = {}
    for name, x in (("q", q32), ("k", k32)):
        codes = np.zeros(x.shape, dtype=np.float64)
        scales = np.zeros((x.shape[0], width), dtype=np.float32)
        for s_, (a, b) in enumerate(bounds):
            if b == a:
                continue
            c, sc = quantize_blocks(x[:, a:b], block)     # tiles aligned to the sequence start
            codes[:, a:b] = c
            scales[:, prefix[s_]:prefix[s_] + sc.shape[1]] = sc
        out[name + "c"], out[name + "s"] = codes, scales
    vc, vs = quantize_blocks(v32, T)
    out["vc"], out["vs"] = vc, vs.reshape(nkv)
    out["cu"] = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    return out


def prefill_fp8_varlen(qz: dict, scale: float, causal: bool = True, block: int = _BLOCK):
    """Packed attention (:func:`attention_ref.prefill_varlen`) on the
    dequantised inputs of :func:`quantize_for_attention_varlen`."""
    cu = qz["cu"]
    prefix = packed_tile_count(cu, block)
    qd = np.zeros(qz["qc"].shape)
    kd = np.zeros(qz["kc"].shape)
    for s_, (a, b) in enumerate(_seq_bounds(cu)):
        if b == a:
            continue
        nt = prefix[s_ + 1] - prefix[s_]
        qd[:, a:b] = dequantize(qz["qc"][:, a:b], qz["qs"][:, prefix[s_]:prefix[s_] + nt], block)
        kd[:, a:b] = dequantize(qz["kc"][:, a:b], qz["ks"][:, prefix[s_]:prefix[s_] + nt], block)
    vd = qz["vc"] * np.asarray(qz["vs"], dtype=np.float64)[:, None, None]
    return prefill_varlen(qd, kd, vd, cu, scale, causal)
