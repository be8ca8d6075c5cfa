"""Python binding of the C ABI in ``include/attn.h``.

Argument marshalling only: shape/dtype checks, output allocation with torch,
raw pointers and the current CUDA stream passed to ``libattn.so``.  Nothing
here computes any part of attention.
"""

from __future__ import annotations

import math
from typing import Optional

import torch

from ._lib import check, lib

_BF16 = torch.bfloat16


# attn_decode_splitkv_ex2 flag (include/attn.h ATTN_DECODE_EARLY_CACHE).
EARLY_CACHE = 1
OUT_BF16 = 1  # ATTN_PREFILL_OUT_BF16


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
            causal: bool = True, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, stream=None, window_left: int = -1,
            softcap: float = 0.0, alibi_slopes: Optional[torch.Tensor] = None,
            out_dtype: torch.dtype = torch.float32):
    """Attention forward over whole sequences (``attn_prefill``; with a
    sliding window, soft-capping or ALiBi slopes ((n_q,) fp32 on the device),
    ``attn_prefill_ex``; with ``out_dtype=torch.bfloat16``,
    ``attn_prefill_ex2`` with ATTN_PREFILL_OUT_BF16).

    q: (B, n_q, N, d) bf16; k, v: (B, n_kv, N, d) bf16.  Returns
    (O (B, n_q, N, d) fp32 or bf16, LSE (B, n_q, N) fp32, natural log).
    """
    _need(q, "q", _BF16, 4)
    _need(k, "k", _BF16, 4)
    _need(v, "v", _BF16, 4)
    B, n_q, N, d = q.shape
    n_kv = k.shape[1]
    if k.shape != (B, n_kv, N, d) or v.shape != k.shape:
        raise ValueError("k and v must be (B, n_kv, N, d) matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype not in (torch.float32, _BF16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((B, n_q, N, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, n_q, N), dtype=torch.float32, device=q.device)
    _need(out, "out", out_dtype, 4)
    _need(lse, "lse", torch.float32, 3)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, n_q, n_kv,
            N, d, float(scale), int(bool(causal)))
    if out_dtype == _BF16:
        al = None
        if alibi_slopes is not None:
            _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
            if alibi_slopes.numel() != n_q:
                raise ValueError("alibi_slopes must have one slope per query head")
            al = alibi_slopes.data_ptr()
        check("attn_prefill_ex2", lib().attn_prefill_ex2(*args, int(window_left), float(softcap),
                                                         al, OUT_BF16, _stream(stream)))
    elif window_left == -1 and softcap == 0.0 and alibi_slopes is None:
        check("attn_prefill", lib().attn_prefill(*args, _stream(stream)))
    else:
        al = None
        if alibi_slopes is not None:
            _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
            if alibi_slopes.numel() != n_q:
                raise ValueError("alibi_slopes must have one slope per query head")
            al = alibi_slopes.data_ptr()
        check("attn_prefill_ex", lib().attn_prefill_ex(*args, int(window_left), float(softcap),
                                                       al, _stream(stream)))
    return out, lse


def prefill_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                   scale: Optional[float] = None, causal: bool = True,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   stream=None, window_left: int = -1, softcap: float = 0.0,
                   alibi_slopes: Optional[torch.Tensor] = None,
                   out_dtype: torch.dtype = torch.float32):
    """Prefill of sequences packed end to end (``attn_prefill_varlen``; with a
    sliding window, soft-capping or ALiBi slopes, ``attn_prefill_varlen_ex``,
    positions counted from each sequence's first row; with
    ``out_dtype=torch.bfloat16``, ``attn_prefill_varlen_ex2``).

    q: (n_q, total, d) bf16; k, v: (n_kv, total, d) bf16; cu_seqlens:
    (num_seqs + 1,) int32 on the device.  Returns (O (n_q, total, d) fp32 or
    bf16, LSE (n_q, total) fp32); rows outside every sequence are left as
    they were in ``out`` / ``lse``.
    """
    _need(q, "q", _BF16, 3)
    _need(k, "k", _BF16, 3)
    _need(v, "v", _BF16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    n_q, T, d = q.shape
    n_kv = k.shape[0]
    if k.shape != (n_kv, T, d) or v.shape != k.shape:
        raise ValueError("k and v must be (n_kv, total, d) matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype not in (torch.float32, _BF16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((n_q, T, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((n_q, T), dtype=torch.float32, device=q.device)
    _need(out, "out", out_dtype, 3)
    _need(lse, "lse", torch.float32, 2)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, T, n_q, n_kv, d, float(scale),
            int(bool(causal)))
    if out_dtype == _BF16:
        al = None
        if alibi_slopes is not None:
            _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
            if alibi_slopes.numel() != n_q:
                raise ValueError("alibi_slopes must have one slope per query head")
            al = alibi_slopes.data_ptr()
        name = "attn_prefill_varlen_ex2"
        st = lib().attn_prefill_varlen_ex2(*args, int(window_left), float(softcap), al, OUT_BF16,
                                           _stream(stream))
    elif window_left != -1 or softcap != 0.0 or alibi_slopes is not None:
        al = None
        if alibi_slopes is not None:
            _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
            if alibi_slopes.numel() != n_q:
                raise ValueError("alibi_slopes must have one slope per query head")
            al = alibi_slopes.data_ptr()
        name = "attn_prefill_varlen_ex"
        st = lib().attn_prefill_varlen_ex(*args, int(window_left), float(softcap), al,
                                          _stream(stream))
    else:
        name = "attn_prefill_varlen"
        st = lib().attn_prefill_varlen(*args, _stream(stream))
    check(name, st)
    return out, lse


def prefill_fp8(q8: torch.Tensor, k8: torch.Tensor, v8t: torch.Tensor, q_scales: torch.Tensor,
                k_scales: torch.Tensor, v_scales: torch.Tensor, scale: float, causal: bool = True,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                stream=None):
    """Prefill on FP8 inputs from :func:`quantize_fp8` (``attn_prefill_fp8``):
    q8 (B, n_q, N, d) and k8 (B, n_kv, N, d) e4m3 codes (uint8), v8t
    (B, n_kv, d, N) transposed, their block / head scales; d is 64 or 128.
    Returns (O (B, n_q, N, d) fp32, LSE (B, n_q, N) fp32)."""
    for t, name in ((q8, "q8"), (k8, "k8"), (v8t, "v8t")):
        _need(t, name, torch.uint8, 4)
    B, n_q, N, d = q8.shape
    n_kv = k8.shape[1]
    if k8.shape != (B, n_kv, N, d) or v8t.shape != (B, n_kv, d, N):
        raise ValueError("k8 must be (B, n_kv, N, d) and v8t (B, n_kv, d, N)")
    for t, name in ((q_scales, "q_scales"), (k_scales, "k_scales"), (v_scales, "v_scales")):
        _need(t, name, torch.float32, t.dim())
    if out is None:
        out = torch.empty((B, n_q, N, d), dtype=torch.float32, device=q8.device)
    if lse is None:
        lse = torch.empty((B, n_q, N), dtype=torch.float32, device=q8.device)
    st = lib().attn_prefill_fp8(q8.data_ptr(), k8.data_ptr(), v8t.data_ptr(), q_scales.data_ptr(),
                                k_scales.data_ptr(), v_scales.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, n_q, n_kv, N, d, float(scale),
                                int(bool(causal)), _stream(stream))
    check("attn_prefill_fp8", st)
    return out, lse


def prefill_fp8_varlen(q8: torch.Tensor, k8: torch.Tensor, v8t: torch.Tensor,
                       q_scales: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                       cu_seqlens: torch.Tensor, scale: float, causal: bool = True,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       stream=None):
    """Packed prefill on FP8 inputs (``attn_prefill_fp8_varlen``): q8 (n_q,
    total, d) and k8 (n_kv, total, d) from :func:`quantize_fp8_varlen`, v8t
    (n_kv, d, total) from :func:`quantize_fp8` (block_rows=0,
    transpose=True), d 64 or 128; every non-empty sequence must start at a
    multiple of 16 rows.  Returns (O (n_q, total, d) fp32, LSE (n_q, total)
    fp32); rows outside every sequence are left as they were in ``out`` /
    ``lse``."""
    for t, name in ((q8, "q8"), (k8, "k8"), (v8t, "v8t")):
        _need(t, name, torch.uint8, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    n_q, T, d = q8.shape
    n_kv = k8.shape[0]
    if k8.shape != (n_kv, T, d) or v8t.shape != (n_kv, d, T):
        raise ValueError("k8 must be (n_kv, total, d) and v8t (n_kv, d, total)")
    for t, name in ((q_scales, "q_scales"), (k_scales, "k_scales"), (v_scales, "v_scales")):
        _need(t, name, torch.float32, t.dim())
    if out is None:
        out = torch.empty((n_q, T, d), dtype=torch.float32, device=q8.device)
    if lse is None:
        lse = torch.empty((n_q, T), dtype=torch.float32, device=q8.device)
    st = lib().attn_prefill_fp8_varlen(q8.data_ptr(), k8.data_ptr(), v8t.data_ptr(),
                                       q_scales.data_ptr(), k_scales.data_ptr(),
                                       v_scales.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, T, n_q,
                                       n_kv, d, float(scale), int(bool(causal)), _stream(stream))
    check("attn_prefill_fp8_varlen", st)
    return out, lse


def quantize_fp8_varlen(x: torch.Tensor, cu_seqlens: torch.Tensor,
                        signs: Optional[torch.Tensor] = None, stream=None):
    """Block quantisation of packed rows (``attn_quantize_fp8_varlen``):
    x (planes, total, d) bf16; each sequence in tiles of 128 rows from its
    first row.  Returns (codes uint8 (planes, total, d), scales fp32
    (planes, ceil(total / 128) + num_seqs)); rows outside every sequence and
    the columns past the last tile are zero."""
    _need(x, "x", _BF16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    planes, T, d = x.shape
    ns = cu_seqlens.numel() - 1
    codes = torch.zeros((planes, T, d), dtype=torch.uint8, device=x.device)
    scales = torch.zeros((planes, -(-T // 128) + ns), dtype=torch.float32, device=x.device)
    sp = None
    if signs is not None:
        _need(signs, "signs", torch.float32, 1)
        if signs.numel() != d:
            raise ValueError("signs must have head_dim entries")
        sp = signs.data_ptr()
    st = lib().attn_quantize_fp8_varlen(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), sp,
                                        cu_seqlens.data_ptr(), ns, T, planes, d, _stream(stream))
    check("attn_quantize_fp8_varlen", st)
    return codes, scales


def quantize_fp8(x: torch.Tensor, signs: Optional[torch.Tensor] = None, block_rows: int = 128,
                 transpose: bool = False, stream=None, codes: Optional[torch.Tensor] = None,
                 scales: Optional[torch.Tensor] = None):
    """FP8 (e4m3) block quantisation with optional incoherent rotation
    (``attn_quantize_fp8``).  x: (..., rows, d) bf16, the leading dimensions
    being planes.  Returns (codes uint8 (planes..., rows, d) or, transposed,
    (planes..., d, rows); scales fp32 (planes..., ceil(rows/128)) or
    (planes...,) when block_rows == 0), written into ``codes`` / ``scales``
    when given (contiguous, of those shapes)."""
    _need(x, "x", _BF16, x.dim())
    lead, rows, d = tuple(x.shape[:-2]), x.shape[-2], x.shape[-1]
    planes = 1
    for n in lead:
        planes *= n
    shape = lead + ((d, rows) if transpose else (rows, d))
    nb = -(-rows // 128)
    sshape = lead + ((nb,) if block_rows else ())
    if codes is None:
        codes = torch.empty(shape, dtype=torch.uint8, device=x.device)
    else:
        _need(codes, "codes", torch.uint8, len(shape))
        if tuple(codes.shape) != shape:
            raise ValueError(f"codes must have shape {shape}")
    if scales is None:
        scales = torch.empty(sshape, dtype=torch.float32, device=x.device)
    else:
        _need(scales, "scales", torch.float32, len(sshape))
        if tuple(scales.shape) != sshape:
            raise ValueError(f"scales must have shape {sshape}")
    sp = None
    if signs is not None:
        _need(signs, "signs", torch.float32, 1)
        if signs.numel() != d:
            raise ValueError("signs must have head_dim entries")
        sp = signs.data_ptr()
    st = lib().attn_quantize_fp8(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), sp, planes,
                                 rows, d, int(block_rows), int(bool(transpose)), _stream(stream))
    check("attn_quantize_fp8", st)
    return codes, scales


def quantize_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     signs: Optional[torch.Tensor] = None, stream=None, out: Optional[tuple] = None):
    """FP8 inputs of :func:`prefill_fp8` for Q, K and V in one call
    (``attn_quantize_fp8_qkv``): Q and K with 128-row block scales and the
    optional rotation, V with one scale per plane, transposed.  q: (...,
    rows, d), k and v: (..., rows, d) bf16.  Returns (q8, k8, v8t, q_scales,
    k_scales, v_scales), written into ``out`` (a tuple of those six tensors)
    when given; equal bit for bit to three :func:`quantize_fp8` calls."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, name, _BF16, q.dim())
    rows, d = q.shape[-2], q.shape[-1]
    if tuple(k.shape) != tuple(v.shape) or k.shape[-2:] != q.shape[-2:]:
        raise ValueError("k and v must match, and share rows and head_dim with q")
    lq, lk = tuple(q.shape[:-2]), tuple(k.shape[:-2])
    pq = pk = 1
    for n in lq:
        pq *= n
    for n in lk:
        pk *= n
    nb = -(-rows // 128)
    shapes = [(lq + (rows, d), torch.uint8), (lk + (rows, d), torch.uint8),
              (lk + (d, rows), torch.uint8), (lq + (nb,), torch.float32),
              (lk + (nb,), torch.float32), (lk, torch.float32)]
    if out is None:
        out = tuple(torch.empty(sh, dtype=dt, device=q.device) for sh, dt in shapes)
    for t, (sh, dt), name in zip(out, shapes, ("q8", "k8", "v8t", "q_scales", "k_scales",
                                               "v_scales")):
        _need(t, name, dt, len(sh))
        if tuple(t.shape) != sh:
            raise ValueError(f"{name} must have shape {sh}")
    sp = None
    if signs is not None:
        _need(signs, "signs", torch.float32, 1)
        if signs.numel() != d:
            raise ValueError("signs must have head_dim entries")
        sp = signs.data_ptr()
    st = lib().attn_quantize_fp8_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     *(t.data_ptr() for t in out), sp, pq, pk, rows, d,
                                     _stream(stream))
    check("attn_quantize_fp8_qkv", st)
    return out


def decode_num_splits(batch: int, n_kv_heads: int, max_kv_len: int, num_sms: int = 0) -> int:
    """The split-count policy (``attn_decode_num_splits``)."""
    return int(lib().attn_decode_num_splits(int(batch), int(n_kv_heads), int(max_kv_len),
                                            int(num_sms)))


def _decode_call(q, k_cache, v_cache, kv_lens, block_table, num_splits, max_kv_len, scale,
                 o_partial, lse_partial, stream, new_kv=None, window_left=-1, softcap=0.0,
                 alibi_slopes=None, early_cache=False):
    """Shape checks and marshalling shared by the plain and appending decode."""
    _need(q, "q", _BF16, 3)
    _need(k_cache, "k_cache", _BF16, 4)
    _need(v_cache, "v_cache", _BF16, 4)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    B, n_q, d = q.shape
    n_kv = k_cache.shape[2]
    if k_cache.shape[3] != d or kv_lens.shape[0] != B:
        raise ValueError("cache head_dim or kv_lens length does not match q")
    if new_kv is not None:
        for t, name in zip(new_kv, ("k_new", "v_new")):
            _need(t, name, _BF16, 3)
            if tuple(t.shape) != (B, n_kv, d):
                raise ValueError(f"{name} must be (batch, n_kv_heads, head_dim)")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        if block_table.shape[0] != B:
            raise ValueError("block_table must have one row per sequence")
        num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
        max_blocks = block_table.shape[1]
        if max_kv_len is None:
            max_kv_len = max_blocks * block_size
        bt_ptr = block_table.data_ptr()
    else:
        if k_cache.shape[0] != B:
            raise ValueError("a contiguous cache must be (B, L, n_kv, d)")
        num_blocks, block_size, max_blocks = 0, 0, 0
        max_kv_len = k_cache.shape[1]
        bt_ptr = None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits == 0:
        num_splits = decode_num_splits(B, n_kv, max_kv_len)
    if o_partial is None:
        o_partial = torch.empty((num_splits, B, n_q, d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((num_splits, B, n_q), dtype=torch.float32, device=q.device)
    _need(o_partial, "o_partial", torch.float32, 4)
    _need(lse_partial, "lse_partial", torch.float32, 3)
    if o_partial.shape[0] != num_splits or lse_partial.shape[0] != num_splits:
        raise ValueError("partial buffers must have num_splits rows")
    tail = (kv_lens.data_ptr(), int(num_splits), o_partial.data_ptr(), lse_partial.data_ptr(), B,
            n_q, n_kv, d, block_size, max_blocks, num_blocks, int(max_kv_len), float(scale),
            _stream(stream))
    variant = window_left != -1 or softcap != 0.0 or alibi_slopes is not None
    al = None
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
        if alibi_slopes.numel() != n_q:
            raise ValueError("alibi_slopes must have one slope per query head")
        al = alibi_slopes.data_ptr()
    if new_kv is None and early_cache:
        name = "attn_decode_splitkv_ex2"
        st = lib().attn_decode_splitkv_ex2(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           bt_ptr, *tail[:-1], int(window_left), float(softcap),
                                           al, EARLY_CACHE, tail[-1])
    elif new_kv is None and variant:
        name = "attn_decode_splitkv_ex"
        st = lib().attn_decode_splitkv_ex(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                          bt_ptr, *tail[:-1], int(window_left), float(softcap),
                                          al, tail[-1])
    elif new_kv is None:
        name = "attn_decode_splitkv"
        st = lib().attn_decode_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), bt_ptr,
                                       *tail)
    elif variant:
        name = "attn_decode_append_splitkv_ex"
        st = lib().attn_decode_append_splitkv_ex(q.data_ptr(), new_kv[0].data_ptr(),
                                                 new_kv[1].data_ptr(), k_cache.data_ptr(),
                                                 v_cache.data_ptr(), bt_ptr, *tail[:-1],
                                                 int(window_left), float(softcap), al, tail[-1])
    else:
        name = "attn_decode_append_splitkv"
        st = lib().attn_decode_append_splitkv(q.data_ptr(), new_kv[0].data_ptr(),
                                              new_kv[1].data_ptr(), k_cache.data_ptr(),
                                              v_cache.data_ptr(), bt_ptr, *tail)
    check(name, st)
    return o_partial, lse_partial


def decode_splitkv(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   kv_lens: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                   num_splits: int = 0, max_kv_len: Optional[int] = None,
                   scale: Optional[float] = None, o_partial: Optional[torch.Tensor] = None,
                   lse_partial: Optional[torch.Tensor] = None, stream=None, window_left: int = -1,
                   softcap: float = 0.0, alibi_slopes: Optional[torch.Tensor] = None,
                   early_cache: bool = False):
    """Split-KV single-token decode (``attn_decode_splitkv``; with a sliding
    window or soft-capping, ``attn_decode_splitkv_ex``; with
    ``early_cache=True``, ``attn_decode_splitkv_ex2`` with
    ATTN_DECODE_EARLY_CACHE: the kernel may start streaming the cache before
    the previous kernel on the stream has finished, which must then write
    none of kv_lens, block_table and the caches).

    q: (B, n_q, d) bf16.  Paged: k_cache, v_cache (num_blocks, block_size,
    n_kv, d) with block_table (B, max_blocks) int32; contiguous (block_table
    None): (B, L, n_kv, d).  kv_lens: (B,) int32 on the device.
    Returns (o_partial (S, B, n_q, d), lse_partial (S, B, n_q)), fp32.
    """
    return _decode_call(q, k_cache, v_cache, kv_lens, block_table, num_splits, max_kv_len, scale,
                        o_partial, lse_partial, stream, window_left=window_left, softcap=softcap,
                        alibi_slopes=alibi_slopes, early_cache=early_cache)


def decode_append_splitkv(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          k_cache: torch.Tensor, v_cache: torch.Tensor, kv_lens: torch.Tensor,
                          block_table: Optional[torch.Tensor] = None, num_splits: int = 0,
                          max_kv_len: Optional[int] = None, scale: Optional[float] = None,
                          o_partial: Optional[torch.Tensor] = None,
                          lse_partial: Optional[torch.Tensor] = None, stream=None,
                          window_left: int = -1, softcap: float = 0.0,
                          alibi_slopes: Optional[torch.Tensor] = None):
    """Split-KV decode that first writes each sequence's new key and value
    (k_new, v_new: (B, n_kv, d) bf16) into the cache at position kv_lens[b]
    and attends over kv_lens[b] + 1 tokens (``attn_decode_append_splitkv``;
    with a sliding window, soft-capping or ALiBi slopes,
    ``attn_decode_append_splitkv_ex``).  kv_lens is not modified: the caller
    increments it afterwards.
    """
    return _decode_call(q, k_cache, v_cache, kv_lens, block_table, num_splits, max_kv_len, scale,
                        o_partial, lse_partial, stream, new_kv=(k_new, v_new),
                        window_left=window_left, softcap=softcap, alibi_slopes=alibi_slopes)


def combine(o_partial: torch.Tensor, lse_partial: torch.Tensor,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    """Merge split partials by their LSE weights (``attn_combine``).

    o_partial: (S, B, n_q, d) fp32; lse_partial: (S, B, n_q) fp32.
    Returns (O (B, n_q, d), LSE (B, n_q)), fp32.
    """
    _need(o_partial, "o_partial", torch.float32, 4)
    _need(lse_partial, "lse_partial", torch.float32, 3)
    S, B, n_q, d = o_partial.shape
    if lse_partial.shape != (S, B, n_q):
        raise ValueError("lse_partial must be (S, B, n_q)")
    if out is None:
        out = torch.empty((B, n_q, d), dtype=torch.float32, device=o_partial.device)
    if lse is None:
        lse = torch.empty((B, n_q), dtype=torch.float32, device=o_partial.device)
    _need(out, "out", torch.float32, 3)
    _need(lse, "lse", torch.float32, 2)
    st = lib().attn_combine(o_partial.data_ptr(), lse_partial.data_ptr(), S, B, n_q, d,
                            out.data_ptr(), lse.data_ptr(), _stream(stream))
    check("attn_combine", st)
    return out, lse


def decode(q, k_cache, v_cache, kv_lens, block_table=None, num_splits: int = 0,
           max_kv_len: Optional[int] = None, scale: Optional[float] = None, stream=None,
           window_left: int = -1, softcap: float = 0.0,
           alibi_slopes: Optional[torch.Tensor] = None):
    """Split-KV decode followed by the combine: returns (O (B, n_q, d), LSE (B, n_q)).
    The variants are those of :func:`decode_splitkv`."""
    op, lp = decode_splitkv(q, k_cache, v_cache, kv_lens, block_table, num_splits, max_kv_len,
                            scale, stream=stream, window_left=window_left, softcap=softcap,
                            alibi_slopes=alibi_slopes)
    return combine(op, lp, stream=stream)


def decode_append(q, k_new, v_new, k_cache, v_cache, kv_lens, block_table=None,
                  num_splits: int = 0, max_kv_len: Optional[int] = None,
                  scale: Optional[float] = None, stream=None, window_left: int = -1,
                  softcap: float = 0.0, alibi_slopes: Optional[torch.Tensor] = None):
    """Decode with append followed by the combine: returns (O, LSE); the new
    rows are in the caches afterwards, kv_lens is left to the caller."""
    op, lp = decode_append_splitkv(q, k_new, v_new, k_cache, v_cache, kv_lens, block_table,
                                   num_splits, max_kv_len, scale, stream=stream,
                                   window_left=window_left, softcap=softcap,
                                   alibi_slopes=alibi_slopes)
    return combine(op, lp, stream=stream)


def check_device_status(stream=None) -> None:
    """Synchronises the stream and raises if a kernel recorded an error."""
    check("attn_check_device_status", lib().attn_check_device_status(_stream(stream)))


def set_wait_timeout_ns(timeout_ns: int) -> int:
    """Sets the bound on any kernel-side wait; returns the previous bound."""
    return int(lib().attn_set_wait_timeout_ns(int(timeout_ns)))


def selftest_bounded_wait(stream=None) -> int:
    """Runs the bounded-wait self-test kernel; returns its attn_status code."""
    return int(lib().attn_selftest_bounded_wait(_stream(stream)))


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   kv_lens: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                   num_splits: int = 0, max_kv_len: Optional[int] = None,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, stream=None):
    """Split-KV decode + combine with the partials in the library's fixed
    device buffer (``attn_decode_noalloc``), for callers that cannot allocate
    device memory on their decode path: pass ``out`` and ``lse`` to allocate
    nothing at all.  Returns (O (B, n_q, d), LSE (B, n_q)), fp32."""
    _need(q, "q", _BF16, 3)
    _need(k_cache, "k_cache", _BF16, 4)
    _need(v_cache, "v_cache", _BF16, 4)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    B, n_q, d = q.shape
    n_kv = k_cache.shape[2]
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        num_blocks, block_size, max_blocks = k_cache.shape[0], k_cache.shape[1], block_table.shape[1]
        if max_kv_len is None:
            max_kv_len = max_blocks * block_size
        bt_ptr = block_table.data_ptr()
    else:
        num_blocks, block_size, max_blocks = 0, 0, 0
        max_kv_len = k_cache.shape[1]
        bt_ptr = None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, n_q, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, n_q), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, 3)
    _need(lse, "lse", torch.float32, 2)
    st = lib().attn_decode_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), bt_ptr,
                                   kv_lens.data_ptr(), int(num_splits), out.data_ptr(),
                                   lse.data_ptr(), B, n_q, n_kv, d, block_size, max_blocks,
                                   num_blocks, int(max_kv_len), float(scale), _stream(stream))
    check("attn_decode_noalloc", st)
    return out, lse
