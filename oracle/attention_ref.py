"""Float64 CPU oracle for exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` leg are the only callers; the CUDA library never
routes through this file and this file imports nothing from the library.

Source of truth: the explainer page "FlashAttention for inference: tiled
prefill and split-KV decoding" (pofe.ai).  Its §"The bottleneck it attacks"
defines standard attention as S = Q K^T / sqrt(d), P = softmax(S), O = P V,
materialising the N x N matrices.  Its §"Toy run: tiling and splitting are
exact" and §"The online softmax, with every symbol defined" state that the
tiled / split-KV methods reach that same result up to rounding order.  So
this oracle is that plain definition, written out in float64 with the score
rows materialised; it contains no online softmax, no tiling of the key axis
and no chunked reduction.  The row blocks below only bound memory: each block
holds every key column its rows may see, so nothing is reordered.

Conventions (readings of the page where it is silent; each is listed with its
reason in the design notes of the repository):

* ``scale`` is a parameter; the workloads pass 1/sqrt(head_dim).
* LSE is the natural log of the sum of exponentials of the *scaled* scores,
  lambda = m + log(l) in the page's notation (§"The online softmax ...").
* Causal prefill (§"Prefill: tiles, loop order and the tensor cores") has
  seq_q == seq_k == N and row i sees keys j <= i.
* Grouped-query attention (§"Decode: a different bottleneck", the GQA
  paragraph): g = n_q / n_kv query heads share one key/value head; query head
  h reads key/value head h // g (consecutive grouping).
* Paged cache (same section, the paged-cache paragraph, and §"Minimal
  implementation"): token t of sequence b lives in physical block
  block_table[b, t // block_size] at slot t % block_size, cache layout
  (num_blocks, block_size, n_kv, d).  A contiguous cache has layout
  (batch, max_kv_len, n_kv, d).
* An empty key set (a zero-length sequence or an empty split) has LSE = -inf
  and O = 0: the plain value of an empty sum.
* Variable-length prefill (§"Interaction with post-trained models", the
  paragraph on packed data and variable-length batches): several sequences
  are packed end to end without padding and none attends to another; the
  packed layout is head-major, q (n_q, total, d), k / v (n_kv, total, d), with
  cu_seqlens (num_seqs + 1) marking where each sequence starts.
* Decode with append (§"Minimal implementation", the decode call against a
  paged cache): the per-sequence length counts the tokens already cached; the
  call writes the new token's key and value at that position, attends over
  length + 1 tokens, and leaves the length to the caller to increment.
"""

from __future__ import annotations

from typing import Iterable, Sequence

import numpy as np

__all__ = [
    "masked_attention",
    "prefill",
    "prefill_rows",
    "gather_sequence",
    "decode",
    "decode_partials",
    "combine",
    "append_token",
    "decode_append",
    "prefill_varlen",
    "prefill_varlen_rows",
]

_ROW_BLOCK = 256


def _f64(x) -> np.ndarray:
    """Exact upcast to float64 (bf16 / fp32 values are representable)."""
    if hasattr(x, "detach"):  # a torch tensor; import-free duck typing
        x = x.detach().to("cpu")
        import torch  # local import: only needed for torch inputs

        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def masked_attention(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray,
                     scale: float, allowed: np.ndarray | None = None, softcap: float = 0.0,
                     bias: np.ndarray | None = None):
    """Plain attention of some query rows against a key/value set.

    s_ij = scale * q_i . k_j   (page §"The bottleneck it attacks": S = QK^T/sqrt d)
    LSE_i = log sum_{j allowed} exp(s_ij)
    O_i   = sum_{j allowed} exp(s_ij - LSE_i) v_j   (= softmax(s_i)^T V)

    ``allowed`` is a boolean (rows, keys) matrix; None means every key.
    A row with no allowed key gets LSE = -inf and O = 0.  With softcap > 0
    the scores are first soft-capped, s -> softcap * tanh(s / softcap) (page
    §"Interaction with post-trained models": logit soft-capping is one of the
    attention variants kernels support).  ``bias`` (rows, keys), if given, is
    added to the (capped) scores: the ALiBi bias of the same section.
    Returns (O (rows, dv), LSE (rows,)), float64.
    """
    q_rows = _f64(q_rows)
    k = _f64(k)
    v = _f64(v)
    r = q_rows.shape[0]
    dv = v.shape[1]
    if r == 0:
        return np.zeros((0, dv)), np.zeros((0,))
    if k.shape[0] == 0:
        return np.zeros((r, dv)), np.full((r,), -np.inf)
    s = scale * (q_rows @ k.T)                      # S, materialised
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    if bias is not None:
        s = s + bias
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1)                               # row max (only for stability)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])                 # exp(-inf) = 0 for masked keys
    z = e.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, z)))
    p = e / np.where(empty, 1.0, z)[:, None]        # P = softmax(S)
    o = p @ v                                       # O = P V
    o[empty] = 0.0
    return o, lse


def _kv_head(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """GQA mapping: query head h reads key/value head h // (n_q / n_kv)."""
    g = n_q_heads // n_kv_heads
    return h // g


def _causal_allowed(r0: int, r1: int, ncols: int) -> np.ndarray:
    """Causal mask for rows r0..r1-1 over keys 0..ncols-1: key j <= row i."""
    rows = np.arange(r0, r1)[:, None]
    cols = np.arange(ncols)[None, :]
    return cols <= rows


def _window_allowed(r0: int, r1: int, ncols: int, causal: bool, window_left: int):
    """Rows r0..r1-1 over keys 0..ncols-1: key j <= row i when causal, and
    j >= i - window_left when a sliding window is set (window_left >= 0);
    None when every key is allowed."""
    if not causal and window_left < 0:
        return None
    rows = np.arange(r0, r1)[:, None]
    cols = np.arange(ncols)[None, :]
    ok = np.ones((r1 - r0, ncols), dtype=bool)
    if causal:
        ok &= cols <= rows
    if window_left >= 0:
        ok &= cols >= rows - window_left
    return ok


def _alibi(slope: float, rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """ALiBi bias: -slope * |i - j| for query position i and key position j
    (for causal attention, j <= i, this is -slope * (i - j))."""
    return -slope * np.abs(rows[:, None] - cols[None, :]).astype(np.float64)


def prefill(q, k, v, scale: float, causal: bool = True, window_left: int = -1,
            softcap: float = 0.0, alibi_slopes=None):
    """Attention forward over whole sequences (the prefill case).

    q: (B, n_q, N, d); k, v: (B, n_kv, N, d).  Returns O (B, n_q, N, d) and
    LSE (B, n_q, N), float64.  Causal: row i sees keys j <= i (page
    §"Prefill: tiles, loop order and the tensor cores").  Sliding window
    (window_left >= 0): row i sees only keys j >= i - window_left; softcap > 0
    soft-caps the scores (page §"Interaction with post-trained models", the
    variants kernels support); alibi_slopes (n_q,) adds -slope_h * |i - j|.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    B, n_q, N, d = q.shape
    n_kv = k.shape[1]
    if n_kv == 0 or n_q % n_kv:
        raise ValueError("n_q must be a positive multiple of n_kv")
    o = np.zeros((B, n_q, N, v.shape[3]))
    lse = np.zeros((B, n_q, N))
    for b in range(B):
        for h in range(n_q):
            kh = _kv_head(h, n_q, n_kv)
            for r0 in range(0, N, _ROW_BLOCK):
                r1 = min(N, r0 + _ROW_BLOCK)
                ncols = r1 if causal else N
                if window_left < 0:
                    allowed = _causal_allowed(r0, r1, ncols) if causal else None
                else:
                    allowed = _window_allowed(r0, r1, ncols, causal, window_left)
                bias = None
                if alibi_slopes is not None:
                    bias = _alibi(float(alibi_slopes[h]), np.arange(r0, r1), np.arange(ncols))
                ob, lb = masked_attention(q[b, h, r0:r1], k[b, kh, :ncols],
                                          v[b, kh, :ncols], scale, allowed, softcap, bias)
                o[b, h, r0:r1] = ob
                lse[b, h, r0:r1] = lb
    return o, lse


def prefill_rows(q, k, v, scale: float, causal: bool,
                 rows: Iterable[tuple[int, int, int]], window_left: int = -1,
                 softcap: float = 0.0, alibi_slopes=None):
    """The same definition as :func:`prefill`, for a sample of (b, h, i) rows.

    Used at sizes where every row would take too long on the CPU.  Returns
    O (len(rows), d) and LSE (len(rows),).
    """
    rows = list(rows)
    n_q = q.shape[1]
    n_kv = k.shape[1]
    N = q.shape[2]
    dv = v.shape[3]
    o = np.zeros((len(rows), dv))
    lse = np.zeros((len(rows),))
    groups: dict = {}
    for idx, (b, h, i) in enumerate(rows):
        groups.setdefault((b, _kv_head(h, n_q, n_kv)), []).append((idx, h, i))
    for (b, kh), members in groups.items():
        kb, vb = _f64(k[b, kh]), _f64(v[b, kh])      # upcast once per (sequence, kv head)
        for idx, h, i in members:
            ncols = i + 1 if causal else N
            lo = max(0, i - window_left) if window_left >= 0 else 0
            bias = None
            if alibi_slopes is not None:
                bias = _alibi(float(alibi_slopes[h]), np.array([i]), np.arange(lo, ncols))
            ob, lb = masked_attention(_f64(q[b, h, i:i + 1]), kb[lo:ncols], vb[lo:ncols], scale,
                                      None, softcap, bias)
            o[idx] = ob[0]
            lse[idx] = lb[0]
    return o, lse


def gather_sequence(cache, block_table, b: int, kv_len: int, kv_head: int,
                    block_size: int):
    """Token-ordered (kv_len, d) keys or values of one sequence and head.

    Paged (block_table given): token t is cache[block_table[b, t // bs],
    t % bs, kv_head] (page §"Decode: a different bottleneck", paged caches;
    §"Minimal implementation" for the layouts).  Contiguous (block_table is
    None): token t is cache[b, t, kv_head].  Only the gathered rows are
    upcast, so a large cache is never copied whole.
    """
    if kv_len == 0:
        return np.zeros((0, cache.shape[-1]))
    t = np.arange(kv_len)
    if block_table is None:
        bidx, slot = np.full_like(t, b), t
    else:
        bt = np.asarray(block_table)
        bidx, slot = bt[b, t // block_size], t % block_size
    if hasattr(cache, "detach"):
        import torch  # local import: only needed for torch inputs

        rows = cache[torch.as_tensor(bidx), torch.as_tensor(slot), kv_head]
        return _f64(rows)
    return _f64(np.asarray(cache)[bidx, slot, kv_head])


def decode(q, k_cache, v_cache, block_table, kv_lens: Sequence[int],
           scale: float, block_size: int = 0, window_left: int = -1, softcap: float = 0.0,
           alibi_slopes=None):
    """Single-token decode: one query row per (sequence, query head) attends
    to every cached token 0..kv_len-1 of its sequence.  The query is the
    sequence's last token, position kv_len - 1, so a sliding window
    (window_left >= 0) keeps tokens kv_len - 1 - window_left .. kv_len - 1;
    softcap > 0 soft-caps the scores; alibi_slopes (n_q,) adds
    -slope_h * (kv_len - 1 - j).

    q: (B, n_q, d).  Returns O (B, n_q, d) and LSE (B, n_q), float64.
    """
    q = _f64(q)
    B, n_q, d = q.shape
    n_kv = k_cache.shape[2]
    o = np.zeros((B, n_q, v_cache.shape[-1]))
    lse = np.zeros((B, n_q))
    for b in range(B):
        L = int(kv_lens[b])
        lo = max(0, L - 1 - window_left) if window_left >= 0 else 0
        for kh in range(n_kv):
            kb = gather_sequence(k_cache, block_table, b, L, kh, block_size)[lo:]
            vb = gather_sequence(v_cache, block_table, b, L, kh, block_size)[lo:]
            heads = [h for h in range(n_q) if _kv_head(h, n_q, n_kv) == kh]
            for h in heads:
                bias = None
                if alibi_slopes is not None:
                    bias = _alibi(float(alibi_slopes[h]), np.array([L - 1]), np.arange(lo, L))
                ob, lb = masked_attention(q[b, h:h + 1], kb, vb, scale, None, softcap, bias)
                o[b, h] = ob[0]
                lse[b, h] = lb[0]
    return o, lse


def decode_partials(q, k_cache, v_cache, block_table, kv_lens: Sequence[int],
                    scale: float, block_size: int,
                    ranges: Sequence[Sequence[tuple[int, int]]], softcap: float = 0.0,
                    alibi_slopes=None):
    """Per-split partial results: the plain definition restricted to each
    split's token range (page §"Decode: a different bottleneck", split-KV).

    ranges[b][s] = (start, end) token range of split s of sequence b.
    Returns o_part (S, B, n_q, d) and lse_part (S, B, n_q); an empty range
    gives o = 0, lse = -inf.
    """
    q = _f64(q)
    B, n_q, d = q.shape
    n_kv = k_cache.shape[2]
    S = len(ranges[0])
    o = np.zeros((S, B, n_q, v_cache.shape[-1]))
    lse = np.full((S, B, n_q), -np.inf)
    for b in range(B):
        L = int(kv_lens[b])
        for kh in range(n_kv):
            kb = gather_sequence(k_cache, block_table, b, L, kh, block_size)
            vb = gather_sequence(v_cache, block_table, b, L, kh, block_size)
            heads = [h for h in range(n_q) if _kv_head(h, n_q, n_kv) == kh]
            for s, (t0, t1) in enumerate(ranges[b]):
                for h in heads:
                    bias = None
                    if alibi_slopes is not None:
                        bias = _alibi(float(alibi_slopes[h]), np.array([L - 1]), np.arange(t0, t1))
                    ob, lb = masked_attention(q[b, h:h + 1], kb[t0:t1], vb[t0:t1],
                                              scale, None, softcap, bias)
                    o[s, b, h] = ob[0]
                    lse[s, b, h] = lb[0]
    return o, lse


def combine(o_parts, lse_parts):
    """Merge partial results by their log-sum-exp weights.

    Page §"The online softmax, with every symbol defined" (the paragraph on
    combining independent partial results) and the ``merge`` rule in
    §"Minimal implementation": with chunk outputs o_k and lambda_k =
    m_k + log l_k,  lambda = log sum_k exp(lambda_k)  and
    o = sum_k exp(lambda_k - lambda) o_k  -- a softmax over the chunk axis.
    Splits with lambda_k = -inf carry zero weight; if every split is empty
    the result is o = 0, lambda = -inf.

    o_parts: (S, ..., d); lse_parts: (S, ...).  Returns (o, lse).
    """
    o_parts = _f64(o_parts)
    lse_parts = _f64(lse_parts)
    mx = lse_parts.max(axis=0)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    w = np.exp(lse_parts - mx_safe[None])           # exp(-inf) = 0
    z = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, mx_safe + np.log(np.where(empty, 1.0, z)))
    w = w / np.where(empty, 1.0, z)[None]
    o = (w[..., None] * o_parts).sum(axis=0)
    o[empty] = 0.0
    return o, lse


def _append_position(kv_len: int) -> int:
    """Where the new token goes: right after the kv_len cached tokens."""
    return kv_len


def append_token(k_cache, v_cache, block_table, kv_lens: Sequence[int], k_new, v_new,
                 block_size: int = 0):
    """Writes each sequence's new key and value row into the cache.

    Page §"Minimal implementation": the decode call takes the cache, the
    block table and the per-sequence count of tokens already cached, and
    appends the new keys and values in place; the caller then increments the
    counts.  k_new, v_new: (B, n_kv, d).  Sequence b's new row goes to token
    position kv_lens[b] (a paged cache maps it through the block table as in
    :func:`gather_sequence`).  Returns copies of the two caches with the rows
    written; raises ValueError when a sequence has no free slot.
    """
    def _copy(c):
        return c.clone() if hasattr(c, "clone") else np.array(c, copy=True)

    kc, vc = _copy(k_cache), _copy(v_cache)
    for b in range(len(kv_lens)):
        t = _append_position(int(kv_lens[b]))
        if block_table is None:
            if not 0 <= t < kc.shape[1]:
                raise ValueError(f"sequence {b}: no free slot at position {t}")
            kc[b, t] = k_new[b]
            vc[b, t] = v_new[b]
        else:
            bt = np.asarray(block_table)
            if not 0 <= t < bt.shape[1] * block_size:
                raise ValueError(f"sequence {b}: no free slot at position {t}")
            blk, slot = int(bt[b, t // block_size]), t % block_size
            kc[blk, slot] = k_new[b]
            vc[blk, slot] = v_new[b]
    return kc, vc


def decode_append(q, k_new, v_new, k_cache, v_cache, block_table, kv_lens: Sequence[int],
                  scale: float, block_size: int = 0, window_left: int = -1,
                  softcap: float = 0.0, alibi_slopes=None):
    """Single-token decode that first appends the token's own key and value
    (page §"Minimal implementation"): the query of sequence b attends over its
    kv_lens[b] cached tokens plus the new one.  The variants (sliding window,
    soft-capping, ALiBi; §"Interaction with post-trained models") are those
    of :func:`decode` over the kv_lens[b] + 1 tokens, the new token being the
    query's own position.

    Returns (O (B, n_q, d), LSE (B, n_q), k_cache', v_cache'), the caches as
    :func:`append_token` leaves them.
    """
    kc, vc = append_token(k_cache, v_cache, block_table, kv_lens, k_new, v_new, block_size)
    o, lse = decode(q, kc, vc, block_table, [int(n) + 1 for n in kv_lens], scale, block_size,
                    window_left=window_left, softcap=softcap, alibi_slopes=alibi_slopes)
    return o, lse, kc, vc


def _seq_bounds(cu_seqlens) -> list:
    """(start, end) of each packed sequence from the cumulative lengths."""
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    if cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and not decrease")
    return list(zip(cu[:-1], cu[1:]))


def prefill_varlen(q, k, v, cu_seqlens, scale: float, causal: bool = True,
                   window_left: int = -1, softcap: float = 0.0, alibi_slopes=None):
    """Prefill of sequences packed end to end (page §"Interaction with
    post-trained models", packed data and variable-length batches: examples
    packed into one sequence must not attend to each other).

    q: (n_q, total, d); k, v: (n_kv, total, d); cu_seqlens: (num_seqs + 1,)
    with sequence s occupying rows [cu[s], cu[s+1]).  Each sequence is the
    prefill of :func:`prefill` on its own rows, with the same variants
    (window, soft cap, ALiBi; positions counted from the sequence's first
    row).  Rows past cu[-1] are not part of any sequence and come back as
    O = 0, LSE = -inf.  Returns O (n_q, total, d) and LSE (n_q, total), float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n_q, total, d = q.shape
    o = np.zeros((n_q, total, v.shape[2]))
    lse = np.full((n_q, total), -np.inf)
    for a, b in _seq_bounds(cu_seqlens):
        if b == a:
            continue
        os_, ls_ = prefill(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], scale, causal,
                           window_left=window_left, softcap=softcap, alibi_slopes=alibi_slopes)
        o[:, a:b] = os_[0]
        lse[:, a:b] = ls_[0]
    return o, lse


def prefill_varlen_rows(q, k, v, cu_seqlens, scale: float, causal: bool,
                        rows: Iterable[tuple[int, int]]):
    """:func:`prefill_varlen` for a sample of (head, packed row) pairs, at
    sizes where every row is too slow.  Returns O (len(rows), d), LSE (len(rows),)."""
    bounds = _seq_bounds(cu_seqlens)
    starts = [a for a, _ in bounds]
    n_q, n_kv = q.shape[0], k.shape[0]
    rows = list(rows)
    o = np.zeros((len(rows), v.shape[2]))
    lse = np.full((len(rows),), -np.inf)
    for idx, (h, i) in enumerate(rows):
        s = int(np.searchsorted(starts, i, side="right")) - 1
        a, b = bounds[s]
        if not a <= i < b:
            continue
        kh = _kv_head(h, n_q, n_kv)
        hi = i + 1 if causal else b
        ob, lb = masked_attention(_f64(q[h, i:i + 1]), _f64(k[kh, a:hi]), _f64(v[kh, a:hi]),
                                  scale, None)
        o[idx], lse[idx] = ob[0], lb[0]
    return o, lse
