"""Pins for the float64 oracle: checks against what the pages and mathematics
fix, none of which re-types the oracle's own formula.

* the worked example printed on "FlashAttention for inference: tiled prefill
  and split-KV decoding", §"A worked example by hand" (tests/golden);
* brute force with scalar loops, ``math.exp`` and ``math.fsum``;
* a library routine: torch's float64 CPU ``scaled_dot_product_attention``;
* closed forms and invariants (q = 0, first row, V = 1, key shift, GQA as
  repeated MHA, paged == contiguous, decode == last prefill row);
* the chunk-combine identity (§"The online softmax, with every symbol
  defined", combining partial results) over random chunkings;
* the page's toy run (§"Toy run: tiling and splitting are exact"), re-created
  here with a test-only tiled prefill and split-KV decode;
* planted mistakes: each mutation of the oracle below must break a pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_ref as ref
from exact_io_aware_order_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

TOL = 1e-13


def _f64(t):
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


# ---------------------------------------------------------------------------
# Test-only restatement of the online softmax update (page §"The online
# softmax ...", reconstructed from the prefill pseudo-code and the worked
# example): m_j = max(m_{j-1}, max s_j); c_j = exp(m_{j-1} - m_j);
# l_j = c_j l_{j-1} + sum exp(s_j - m_j); o~_j = c_j o~_{j-1} + sum exp(s_j - m_j) v_j.
# ---------------------------------------------------------------------------

def _online_blocks(scores, values, block):
    """Returns the per-block trace [(m, c, l, otilde)] and final (o, lse)."""
    m, l, ot = -math.inf, 0.0, np.zeros(values.shape[1:])
    trace = []
    for b0 in range(0, len(scores), block):
        s = np.asarray(scores[b0:b0 + block], np.float64)
        vb = np.asarray(values[b0:b0 + block], np.float64)
        m_new = max(m, float(s.max()))
        c = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        l = c * l + p.sum()
        ot = c * ot + (p[:, None] * vb).sum(0) if vb.ndim == 2 else c * ot + (p * vb).sum()
        m = m_new
        trace.append((m, c, l, np.array(ot, copy=True)))
    return trace, ot / l, m + math.log(l)


# ---------------------------------------------------------------------------
# Worked example.
# ---------------------------------------------------------------------------

def test_worked_example_direct(golden):
    g = golden("worked_example.txt")
    s = np.array(g["scores"])
    v = np.array(g["values"])[:, None]
    # d = 1, q = 1, k = s, scale = 1 makes the scores exactly s.
    o, lse = oracle.masked_attention(np.ones((1, 1)), s[:, None], v, 1.0)
    assert abs(o[0, 0] - g["result_o"]) <= 0.5e-4
    assert abs(math.exp(lse[0]) - g["exp_sum"]) <= 0.5e-3
    assert np.allclose(np.exp(s), g["exp_scores"], atol=0.5e-3)


def test_worked_example_blocks_and_combine(golden):
    g = golden("worked_example.txt")
    s = np.array(g["scores"])
    v = np.array(g["values"])
    trace, o, lse = _online_blocks(s, v, 2)
    (m1, _, l1, ot1), (m2, c2, l2, ot2) = trace
    assert m1 == g["block1_m"] and m2 == g["block2_m"]
    assert abs(l1 - g["block1_l"]) <= 0.5e-4
    assert abs(float(ot1) - g["block1_otilde"]) <= 0.5e-4
    assert abs(float(ot1) / l1 - g["block1_interim"]) <= 0.5e-4
    assert abs(c2 - g["block2_c"]) <= 0.5e-4
    assert abs(l2 - g["block2_l"]) <= 0.5e-4
    assert abs(float(ot2) - g["block2_otilde"]) <= 0.5e-4
    assert abs(float(o) - g["result_o"]) <= 0.5e-4
    # The oracle's per-block results merged by its combine rule give the same
    # answer as the oracle on the whole row.
    parts = [oracle.masked_attention(np.ones((1, 1)), s[i:i + 2, None], v[i:i + 2, None], 1.0)
             for i in (0, 2)]
    oc, lc = oracle.combine(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    ow, lw = oracle.masked_attention(np.ones((1, 1)), s[:, None], v[:, None], 1.0)
    assert abs(oc[0, 0] - g["result_o"]) <= 0.5e-4
    assert abs(oc[0, 0] - ow[0, 0]) <= TOL and abs(lc[0] - lw[0]) <= TOL
    assert abs(lse - lw[0]) <= TOL


# ---------------------------------------------------------------------------
# Brute force: scalar loops with math.exp / math.fsum.
# ---------------------------------------------------------------------------

def _brute_prefill(q, k, v, scale, causal, window_left=-1, softcap=0.0, slopes=None):
    B, nq, N, d = q.shape
    nkv = k.shape[1]
    g = nq // nkv
    o = np.zeros(q.shape)
    lse = np.zeros((B, nq, N))
    for b in range(B):
        for h in range(nq):
            kh = h // g
            for i in range(N):
                js = range(i + 1) if causal else range(N)
                if window_left >= 0:
                    js = [j for j in js if j >= i - window_left]
                sc = [scale * math.fsum(q[b, h, i, t] * k[b, kh, j, t] for t in range(d)) for j in js]
                if softcap > 0:
                    sc = [softcap * math.tanh(x / softcap) for x in sc]
                if slopes is not None:
                    sc = [x - slopes[h] * abs(i - j) for x, j in zip(sc, js)]
                m = max(sc)
                z = math.fsum(math.exp(x - m) for x in sc)
                lse[b, h, i] = m + math.log(z)
                for t in range(d):
                    o[b, h, i, t] = math.fsum(math.exp(x - lse[b, h, i]) * v[b, kh, j, t]
                                              for x, j in zip(sc, js))
    return o, lse


def _pin_bruteforce():
    worst = 0.0
    for (B, nq, nkv, N, d, causal) in [(1, 1, 1, 1, 4, True), (1, 2, 1, 2, 3, True),
                                       (2, 2, 2, 3, 8, True), (1, 4, 2, 5, 8, False),
                                       (1, 3, 1, 17, 5, True), (1, 2, 2, 33, 8, True),
                                       (1, 2, 1, 17, 8, False)]:
        x = W.make_prefill(B, nq, nkv, N, d, seed=N + d)
        q, k, v = _f64(x.q), _f64(x.k), _f64(x.v)
        ob, lb = _brute_prefill(q, k, v, x.scale, causal)
        oo, lo = oracle.prefill(x.q, x.k, x.v, x.scale, causal)
        worst = max(worst, np.abs(ob - oo).max(), np.abs(lb - lo).max())
    return worst


def test_bruteforce_tiny_shapes():
    assert _pin_bruteforce() <= TOL


# ---------------------------------------------------------------------------
# Library routine: torch float64 SDPA (GQA expressed by repeating K/V).
# ---------------------------------------------------------------------------

def _pin_sdpa():
    worst = 0.0
    for (B, nq, nkv, N, d, causal) in [(1, 4, 2, 300, 64, True), (2, 6, 3, 129, 32, False),
                                       (1, 7, 1, 200, 128, True)]:
        x = W.make_prefill(B, nq, nkv, N, d, seed=7)
        g = nq // nkv
        q = x.q.double()
        k = x.k.double().repeat_interleave(g, dim=1)
        v = x.v.double().repeat_interleave(g, dim=1)
        ref_o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=causal, scale=x.scale).numpy()
        oo, lo = oracle.prefill(x.q, x.k, x.v, x.scale, causal)
        worst = max(worst, np.abs(ref_o - oo).max())
        # LSE through scipy's logsumexp over the masked score matrix.
        from scipy.special import logsumexp
        sc = (q @ k.transpose(-1, -2)).numpy() * x.scale
        if causal:
            sc = np.where(np.tril(np.ones((N, N), bool)), sc, -np.inf)
        worst = max(worst, np.abs(logsumexp(sc, axis=-1) - lo).max())
    return worst


def test_library_sdpa_float64():
    assert _pin_sdpa() <= 1e-12


# ---------------------------------------------------------------------------
# Closed forms and invariants.
# ---------------------------------------------------------------------------

def _pin_closed_forms():
    worst = 0.0
    x = W.make_prefill(1, 2, 1, 70, 16, seed=3)
    N = 70
    # q = 0: every score is 0, LSE_i = ln(i+1), O_i = mean(v_0..v_i).
    q0 = torch.zeros_like(x.q)
    o, lse = oracle.prefill(q0, x.k, x.v, x.scale, True)
    v = _f64(x.v)[0, 0]
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    worst = max(worst, np.abs(lse[0, 0] - np.log(np.arange(1, N + 1))).max(),
                np.abs(o[0, 1] - prefix_mean).max())
    # Row 0 of causal prefill: O_0 = v_0, LSE_0 = s_00.
    o, lse = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    s00 = x.scale * math.fsum(_f64(x.q)[0, 0, 0] * _f64(x.k)[0, 0, 0])
    worst = max(worst, np.abs(o[0, 0, 0] - v[0]).max(), abs(lse[0, 0, 0] - s00))
    # V = 1 gives O = 1.
    o1, _ = oracle.prefill(x.q, x.k, torch.ones_like(x.v), x.scale, True)
    worst = max(worst, np.abs(o1 - 1.0).max())
    # Adding c to every key leaves O unchanged and shifts LSE_i by scale q_i.c.
    c = torch.linspace(-0.5, 0.5, 16, dtype=torch.float64)
    ks = x.k.double() + c
    o2, lse2 = oracle.prefill(x.q, ks, x.v, x.scale, True)
    shift = x.scale * (_f64(x.q) @ c.numpy())
    worst = max(worst, np.abs(o2 - o).max() / 1e2, np.abs(lse2 - lse - shift).max() / 1e2)
    return worst


def test_closed_forms():
    assert _pin_closed_forms() <= TOL


def _pin_gqa():
    """GQA equals MHA with each kv head repeated g times (consecutive groups)."""
    x = W.make_prefill(1, 6, 2, 40, 8, seed=5)
    o, lse = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    om, lm = oracle.prefill(x.q, x.k.repeat_interleave(3, dim=1),
                            x.v.repeat_interleave(3, dim=1), x.scale, True)
    return max(np.abs(o - om).max(), np.abs(lse - lm).max())


def test_gqa_is_repeated_mha():
    assert _pin_gqa() <= TOL


def test_decode_equals_last_prefill_row_and_paged_equals_contiguous():
    N, nq, nkv, d = 97, 4, 2, 16
    x = W.make_prefill(1, nq, nkv, N, d, seed=11)
    op, lp = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    # Contiguous cache (B, L, n_kv, d) holding the same keys/values.
    kc = x.k[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    vc = x.v[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    q = x.q[:, :, N - 1]
    od, ld = oracle.decode(q, kc, vc, None, [N], x.scale)
    assert np.abs(od - op[:, :, N - 1]).max() <= TOL
    assert np.abs(ld - lp[:, :, N - 1]).max() <= TOL
    # The same tokens laid out in a paged cache through a permuted block table.
    bs = 8
    nb = (N + bs - 1) // bs
    perm = torch.randperm(nb + 3, generator=torch.Generator().manual_seed(2))
    kp = torch.zeros(nb + 3, bs, nkv, d, dtype=torch.float64)
    vp = torch.zeros_like(kp)
    table = torch.zeros(1, nb, dtype=torch.int32)
    for j in range(nb):
        t0, t1 = j * bs, min(N, (j + 1) * bs)
        kp[perm[j], :t1 - t0] = kc[0, t0:t1].double()
        vp[perm[j], :t1 - t0] = vc[0, t0:t1].double()
        table[0, j] = int(perm[j])
    # Slots past the last token hold NaN: they must never be read.
    kp[perm[nb - 1], N - (nb - 1) * bs:] = float("nan")
    vp[perm[nb - 1], N - (nb - 1) * bs:] = float("nan")
    og, lg = oracle.decode(q, kp, vp, table, [N], x.scale, bs)
    assert np.abs(og - od).max() <= TOL and np.abs(lg - ld).max() <= TOL


def test_empty_sequence_and_empty_split():
    x = W.make_decode_contiguous(2, 4, 2, 16, 5, seed=1)
    lens = [0, 5]
    o, lse = oracle.decode(x.q, x.k_cache, x.v_cache, None, lens, x.scale)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
    ranges = [[(0, 0), (0, 0)], [(0, 3), (3, 3)]]
    op, lp = oracle.decode_partials(x.q, x.k_cache, x.v_cache, None, lens, x.scale, 0, ranges)
    assert np.all(np.isneginf(lp[:, 0])) and np.all(op[:, 0] == 0)
    assert np.all(np.isneginf(lp[1, 1])) and np.all(op[1, 1] == 0)
    oc, lc = oracle.combine(op, lp)
    assert np.all(oc[0] == 0.0) and np.all(np.isneginf(lc[0]))


# ---------------------------------------------------------------------------
# Attention variants (page §"Interaction with post-trained models": sliding
# windows and logit soft-capping are among the variants kernels support).
# ---------------------------------------------------------------------------

def _pin_variants():
    """Sliding window and soft-capping against scalar brute force (math.tanh,
    math.fsum), causal and not, GQA."""
    rng = np.random.default_rng(17)
    worst = 0.0
    for N, nq, nkv, d, causal, W, cap in [(19, 2, 1, 4, True, 3, 0.0), (23, 4, 2, 8, True, 0, 0.0),
                                          (17, 2, 2, 4, False, 5, 0.0), (21, 4, 1, 8, True, -1, 1.5),
                                          (16, 2, 1, 4, True, 6, 2.0), (13, 2, 2, 8, False, -1, 0.7)]:
        q = rng.standard_normal((1, nq, N, d)) * 2
        k = rng.standard_normal((1, nkv, N, d))
        v = rng.standard_normal((1, nkv, N, d))
        ob, lb = _brute_prefill(q, k, v, 0.9, causal, W, cap)
        oo, lo = oracle.prefill(q, k, v, 0.9, causal, window_left=W, softcap=cap)
        worst = max(worst, float(np.abs(ob - oo).max()), float(np.abs(lb - lo).max()))
    # ALiBi, with and without a window, causal and not
    for N, nq, nkv, d, causal, W in [(18, 4, 2, 4, True, -1), (15, 2, 1, 8, False, -1),
                                     (20, 4, 4, 4, True, 5)]:
        q = rng.standard_normal((1, nq, N, d))
        k = rng.standard_normal((1, nkv, N, d))
        v = rng.standard_normal((1, nkv, N, d))
        slopes = [2.0 ** (-8.0 * (h + 1) / nq) for h in range(nq)]
        ob, lb = _brute_prefill(q, k, v, 0.7, causal, W, 0.0, slopes)
        oo, lo = oracle.prefill(q, k, v, 0.7, causal, window_left=W, alibi_slopes=slopes)
        worst = max(worst, float(np.abs(ob - oo).max()), float(np.abs(lb - lo).max()))
    return worst


def test_variants_brute_force():
    assert _pin_variants() <= TOL


def test_variant_closed_forms_and_limits():
    x = W.make_prefill(1, 4, 2, 300, 16, seed=2)
    q, k, v = x.q, x.k, x.v
    # window 0: every row sees only itself -> O_i = v_i, LSE_i = s_ii
    o, lse = oracle.prefill(q, k, v, x.scale, True, window_left=0)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for h in range(4):
        assert np.abs(o[0, h] - vd[0, h // 2]).max() <= TOL
        sii = x.scale * np.einsum("nd,nd->n", qd[0, h], kd[0, h // 2])
        assert np.abs(lse[0, h] - sii).max() <= TOL
    # a window covering the whole sequence changes nothing
    o_full, l_full = oracle.prefill(q, k, v, x.scale, True)
    o_w, l_w = oracle.prefill(q, k, v, x.scale, True, window_left=299)
    assert np.abs(o_w - o_full).max() <= TOL and np.abs(l_w - l_full).max() <= TOL
    # soft-capping with a huge cap is the identity on the scores (tanh(u) = u - u^3/3 + ...)
    o_c, l_c = oracle.prefill(q, k, v, x.scale, True, softcap=1e7)
    assert np.abs(o_c - o_full).max() <= 1e-10 and np.abs(l_c - l_full).max() <= 1e-10
    # rows sampled one by one agree with whole prefill, window + cap
    o_v, l_v = oracle.prefill(q, k, v, x.scale, True, window_left=40, softcap=3.0)
    rows = [(0, 0, 0), (0, 3, 41), (0, 1, 299), (0, 2, 120)]
    orow, lrow = oracle.prefill_rows(q, k, v, x.scale, True, rows, window_left=40, softcap=3.0)
    for idx, (b, h, i) in enumerate(rows):
        assert np.abs(orow[idx] - o_v[b, h, i]).max() <= TOL and abs(lrow[idx] - l_v[b, h, i]) <= TOL


def test_decode_variants_equal_last_prefill_row():
    N = 211
    x = W.make_prefill(1, 6, 2, N, 16, seed=8)
    kc = x.k[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    vc = x.v[0].permute(1, 0, 2).unsqueeze(0).contiguous()
    slopes = [0.5, 0.25, 0.125, 0.0625, 0.03125, 0.0]
    for Wl, cap, al in [(50, 0.0, None), (-1, 2.5, None), (7, 1.0, None), (0, 0.0, None),
                        (-1, 0.0, slopes), (30, 0.0, slopes)]:
        op, lp = oracle.prefill(x.q, x.k, x.v, x.scale, True, window_left=Wl, softcap=cap,
                                alibi_slopes=al)
        od, ld = oracle.decode(x.q[:, :, N - 1], kc, vc, None, [N], x.scale, window_left=Wl,
                               softcap=cap, alibi_slopes=al)
        assert np.abs(od - op[:, :, N - 1]).max() <= TOL
        assert np.abs(ld - lp[:, :, N - 1]).max() <= TOL


# ---------------------------------------------------------------------------
# Decode with append (page §"Minimal implementation": the decode call writes
# the new token's key and value at position cache_seqlens[b], attends over
# cache_seqlens[b] + 1 tokens; the caller increments the lengths).
# ---------------------------------------------------------------------------

def _paged_empty_cache(n_blocks_used, extra, bs, nkv, d, seed):
    perm = torch.randperm(n_blocks_used + extra, generator=torch.Generator().manual_seed(seed))
    table = perm[:n_blocks_used].to(torch.int32).reshape(1, -1)
    kc = torch.full((n_blocks_used + extra, bs, nkv, d), float("nan"), dtype=torch.float64)
    return table, kc, kc.clone()


def _pin_append():
    """Token-by-token decode with append, starting from an empty cache full
    of NaN, reproduces every row of causal prefill (an independently pinned
    definition): paged with a permuted block table, and contiguous."""
    N, nq, nkv, d, bs = 37, 4, 2, 8, 8
    x = W.make_prefill(1, nq, nkv, N, d, seed=5)
    op, lp = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    table, kc, vc = _paged_empty_cache((N + bs - 1) // bs, 2, bs, nkv, d, seed=3)
    kk = torch.full((1, N + 3, nkv, d), float("nan"), dtype=torch.float64)  # spare slots
    vv = kk.clone()
    err = 0.0
    for t in range(N):
        q, kn, vn = x.q[:, :, t], x.k[:, :, t], x.v[:, :, t]
        o, lse, kc, vc = oracle.decode_append(q, kn, vn, kc, vc, table, [t], x.scale, bs)
        o2, lse2, kk, vv = oracle.decode_append(q, kn, vn, kk, vv, None, [t], x.scale)
        for oo, ll in ((o, lse), (o2, lse2)):
            err = max(err, float(np.abs(oo - op[:, :, t]).max()), float(np.abs(ll - lp[:, :, t]).max()))
    return err


def test_decode_append_reproduces_prefill_rows():
    assert _pin_append() <= TOL


def test_decode_append_with_variants_reproduces_prefill_rows():
    """Token-by-token decode with append under a sliding window, soft-capping
    or ALiBi, from an empty paged cache, reproduces every row of causal
    prefill under the same variant (the prefill being pinned on its own)."""
    N, nq, nkv, d, bs = 29, 4, 2, 8, 8
    x = W.make_prefill(1, nq, nkv, N, d, seed=6)
    slopes = [0.5, 0.25, 0.125, 0.0625]
    for Wl, cap, al in [(5, 0.0, None), (-1, 1.5, None), (3, 2.0, None), (-1, 0.0, slopes),
                        (6, 0.0, slopes)]:
        op, lp = oracle.prefill(x.q, x.k, x.v, x.scale, True, window_left=Wl, softcap=cap,
                                alibi_slopes=al)
        table, kc, vc = _paged_empty_cache((N + bs - 1) // bs, 1, bs, nkv, d, seed=4)
        for t in range(N):
            o, lse, kc, vc = oracle.decode_append(x.q[:, :, t], x.k[:, :, t], x.v[:, :, t], kc, vc,
                                                  table, [t], x.scale, bs, window_left=Wl,
                                                  softcap=cap, alibi_slopes=al)
            assert np.abs(o - op[:, :, t]).max() <= TOL, (Wl, cap, al is not None, t)
            assert np.abs(lse - lp[:, :, t]).max() <= TOL


def test_decode_append_closed_form_and_written_slot():
    """kv_len = 0: the query sees only its own token, so O = v_new of its kv
    head and LSE = scale * q . k_new.  Exactly one slot per sequence changes."""
    B, nq, nkv, d, bs = 2, 6, 3, 16, 4
    g = nq // nkv
    gen = torch.Generator().manual_seed(9)
    q = torch.randn(B, nq, d, generator=gen, dtype=torch.float64)
    kn = torch.randn(B, nkv, d, generator=gen, dtype=torch.float64)
    vn = torch.randn(B, nkv, d, generator=gen, dtype=torch.float64)
    table = torch.tensor([[3, 1], [0, 2]], dtype=torch.int32)
    kc = torch.randn(4, bs, nkv, d, generator=gen, dtype=torch.float64)
    vc = torch.randn(4, bs, nkv, d, generator=gen, dtype=torch.float64)
    o, lse, kc2, vc2 = oracle.decode_append(q, kn, vn, kc, vc, table, [0, 5], 0.3, bs)
    for h in range(nq):
        assert np.abs(o[0, h] - vn[0, h // g].numpy()).max() <= TOL
        assert abs(lse[0, h] - 0.3 * float(q[0, h] @ kn[0, h // g])) <= TOL
    changed = (kc2 != kc).any(dim=(2, 3)) | (vc2 != vc).any(dim=(2, 3))
    assert changed.sum() == 2 and changed[3, 0] and changed[2, 1]   # seq 0 -> block 3 slot 0,
    assert torch.equal(kc2[2, 1], kn[1]) and torch.equal(vc2[3, 0], vn[0])  # seq 1 -> pos 5
    # the caller's caches are not modified
    assert not torch.equal(kc2, kc)


def test_decode_append_full_cache_raises():
    x = W.make_decode_contiguous(1, 2, 1, 8, 16, seed=1, max_kv_len=16)
    with pytest.raises(ValueError):
        oracle.decode_append(x.q, x.k_cache[:, 0], x.v_cache[:, 0], x.k_cache, x.v_cache, None,
                             [16], x.scale)


# ---------------------------------------------------------------------------
# Variable-length (packed) prefill (page §"Interaction with post-trained
# models": packed examples must not attend to each other).
# ---------------------------------------------------------------------------

def _pin_varlen():
    """Packed prefill against an independent formulation: ONE masked
    attention over the whole packed sequence with the block-diagonal causal
    mask (same sequence and j <= i), and against brute force on a tiny case."""
    lens = [5, 1, 0, 17, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, nq, nkv, d = int(cu[-1]) + 3, 4, 2, 8          # 3 rows past the last sequence
    g = torch.Generator().manual_seed(13)
    q = torch.randn(nq, T, d, generator=g, dtype=torch.float64)
    k = torch.randn(nkv, T, d, generator=g, dtype=torch.float64)
    v = torch.randn(nkv, T, d, generator=g, dtype=torch.float64)
    seq = np.full(T, -1)
    for s_, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        seq[a:b] = s_
    err = 0.0
    for causal in (True, False):
        o, lse = oracle.prefill_varlen(q, k, v, cu, 0.37, causal)
        allowed = (seq[:, None] == seq[None, :]) & (seq[:, None] >= 0)
        if causal:
            allowed &= np.arange(T)[None, :] <= np.arange(T)[:, None]
        for h in range(nq):
            ob, lb = ref.masked_attention(q[h].numpy(), k[h // (nq // nkv)].numpy(),
                                          v[h // (nq // nkv)].numpy(), 0.37, allowed)
            fin = np.isfinite(lb)
            if not np.array_equal(fin, np.isfinite(lse[h])):
                return math.inf                       # an empty row where there is none, or back
            err = max(err, float(np.abs(ob - o[h]).max()), float(np.abs(lb[fin] - lse[h][fin]).max()))
        # brute force on one row of each non-empty sequence
        for a, b in zip(cu[:-1], cu[1:]):
            if b == a:
                continue
            i = b - 1
            for h in (0, nq - 1):
                kh = h // (nq // nkv)
                hi = i + 1 if causal else b
                sc = [0.37 * math.fsum(float(q[h, i, t]) * float(k[kh, j, t]) for t in range(d))
                      for j in range(a, hi)]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                z = math.fsum(w)
                bo = [math.fsum(w[jj] * float(v[kh, a + jj, t]) for jj in range(len(w))) / z
                      for t in range(d)]
                err = max(err, max(abs(bo[t] - o[h, i, t]) for t in range(d)),
                          abs(mx + math.log(z) - lse[h, i]))
    return err


def test_varlen_prefill_matches_block_diagonal_mask_and_brute_force():
    assert _pin_varlen() <= TOL


def _pin_varlen_variants():
    """Packed prefill with a window, a soft cap or ALiBi against scalar brute
    force on each sequence's own rows (positions counted from the sequence's
    first row); rows past the last sequence stay O = 0, LSE = -inf."""
    lens = [7, 0, 12, 5]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, nq, nkv, d = int(cu[-1]) + 2, 4, 2, 8
    rng = np.random.default_rng(23)
    q = rng.standard_normal((nq, T, d)) * 1.5
    k = rng.standard_normal((nkv, T, d))
    v = rng.standard_normal((nkv, T, d))
    slopes = [2.0 ** (-8.0 * (h + 1) / nq) for h in range(nq)]
    worst = 0.0
    for causal, W, cap, sl in [(True, 3, 0.0, None), (False, 4, 0.0, None), (True, -1, 1.3, None),
                               (False, 2, 0.9, None), (True, -1, 0.0, slopes),
                               (False, 5, 0.0, slopes)]:
        o, lse = oracle.prefill_varlen(q, k, v, cu, 0.8, causal, window_left=W, softcap=cap,
                                       alibi_slopes=sl)
        for a, b in zip(cu[:-1], cu[1:]):
            if b == a:
                continue
            ob, lb = _brute_prefill(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], 0.8, causal,
                                    W, cap, sl)
            worst = max(worst, float(np.abs(ob[0] - o[:, a:b]).max()),
                        float(np.abs(lb[0] - lse[:, a:b]).max()))
        if not (np.all(o[:, cu[-1]:] == 0) and np.all(np.isneginf(lse[:, cu[-1]:]))):
            return math.inf
    return worst


def test_varlen_variants_brute_force():
    assert _pin_varlen_variants() <= TOL


def test_varlen_sampled_rows_match_full():
    lens = [130, 7, 300]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = W.make_prefill(1, 4, 2, int(cu[-1]), 16, seed=4)
    q, k, v = x.q[0], x.k[0], x.v[0]
    o, lse = oracle.prefill_varlen(q, k, v, cu, x.scale, True)
    rows = [(0, 0), (3, 129), (1, 130), (2, 136), (0, 137), (3, 436)]
    orow, lrow = oracle.prefill_varlen_rows(q, k, v, cu, x.scale, True, rows)
    for idx, (h, i) in enumerate(rows):
        assert np.abs(orow[idx] - o[h, i]).max() <= TOL and abs(lrow[idx] - lse[h, i]) <= TOL


# ---------------------------------------------------------------------------
# Chunk-combine identity.
# ---------------------------------------------------------------------------

def _pin_combine():
    """Combine identity (page "FlashAttention for inference", section "The online
    softmax, with every symbol defined", combining partial results): merging the
    per-chunk partials of any chunking, empty chunks included, gives the whole
    row's output and LSE -- plain, soft-capped and with ALiBi (the partials of
    a variant are that variant's definition restricted to the chunk)."""
    rng = np.random.default_rng(0)
    worst = 0.0
    x = W.make_decode_contiguous(1, 6, 2, 32, 300, seed=4)
    slopes = [2.0 ** (-8.0 * (h + 1) / 6) for h in range(6)]
    cases = [{}, {"softcap": 0.8}, {"alibi_slopes": slopes}]
    for kw in cases:
        o_full, l_full = oracle.decode(x.q, x.k_cache, x.v_cache, None, [300], x.scale, **kw)
        for trial in range(6):
            cuts = np.sort(rng.choice(np.arange(0, 301), size=rng.integers(1, 7), replace=True))
            bounds = [0] + cuts.tolist() + [300]
            ranges = [[(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)] + [(0, 0)]]
            op, lp = oracle.decode_partials(x.q, x.k_cache, x.v_cache, None, [300], x.scale, 0,
                                            ranges, **kw)
            oc, lc = oracle.combine(op, lp)
            worst = max(worst, np.abs(oc - o_full).max(), np.abs(lc - l_full).max())
            perm = rng.permutation(op.shape[0])           # order of chunks is irrelevant
            oc2, lc2 = oracle.combine(op[perm], lp[perm])
            worst = max(worst, np.abs(oc2 - oc).max(), np.abs(lc2 - lc).max())
    return worst


def _pin_partials_bruteforce():
    """Each split's partial (o, lse), plain and with each variant, against
    scalar brute force (math.exp, math.tanh, math.fsum) over that split's
    tokens only: the query is at position kv_len - 1, so ALiBi's distance is
    kv_len - 1 - j whatever split holds token j."""
    rng = np.random.default_rng(23)
    nq, nkv, d, L = 4, 2, 4, 29
    q = rng.standard_normal((1, nq, d))
    kc = rng.standard_normal((1, L, nkv, d))
    vc = rng.standard_normal((1, L, nkv, d))
    ranges = [[(0, 7), (7, 7), (7, 20), (20, 29)]]
    slopes = [0.3, 0.05, 0.7, 0.11]
    worst = 0.0
    for cap, sl in ((0.0, None), (1.3, None), (0.0, slopes)):
        op, lp = oracle.decode_partials(q, kc, vc, None, [L], 0.8, 0, ranges, softcap=cap,
                                        alibi_slopes=sl)
        for s, (t0, t1) in enumerate(ranges[0]):
            for h in range(nq):
                kh = h // (nq // nkv)
                sc = [0.8 * math.fsum(q[0, h, t] * kc[0, j, kh, t] for t in range(d))
                      for j in range(t0, t1)]
                if cap > 0:
                    sc = [cap * math.tanh(v_ / cap) for v_ in sc]
                if sl is not None:
                    sc = [v_ - sl[h] * (L - 1 - j) for v_, j in zip(sc, range(t0, t1))]
                if not sc:
                    worst = max(worst, float(np.abs(op[s, 0, h]).max()),
                                0.0 if lp[s, 0, h] == -np.inf else math.inf)
                    continue
                m = max(sc)
                lse = m + math.log(math.fsum(math.exp(v_ - m) for v_ in sc))
                o = [math.fsum(math.exp(v_ - lse) * vc[0, j, kh, t]
                               for v_, j in zip(sc, range(t0, t1))) for t in range(d)]
                worst = max(worst, abs(lse - lp[s, 0, h]), float(np.abs(np.array(o) - op[s, 0, h]).max()))
    return worst


def test_partials_with_variants_brute_force():
    assert _pin_partials_bruteforce() <= TOL


def test_combine_identity_random_chunkings():
    assert _pin_combine() <= TOL


def test_combine_matches_softmax_over_chunks_rule():
    """The page's merge rule: weights = softmax of the LSEs over the chunk axis."""
    rng = np.random.default_rng(1)
    o_parts = rng.standard_normal((5, 3, 7))
    lse_parts = rng.standard_normal((5, 3)) * 4
    w = torch.softmax(torch.as_tensor(lse_parts), dim=0).numpy()
    o, lse = oracle.combine(o_parts, lse_parts)
    assert np.abs(o - (w[..., None] * o_parts).sum(0)).max() <= TOL
    assert np.abs(lse - torch.logsumexp(torch.as_tensor(lse_parts), 0).numpy()).max() <= TOL


# ---------------------------------------------------------------------------
# The page's toy run, re-created with test-only tiled / split restatements.
# ---------------------------------------------------------------------------

def _tiled_prefill_head(q, k, v, scale, tile):
    """FA-2 loop order with the online softmax, causal, float64 (test-only)."""
    N, d = q.shape
    o = np.zeros((N, d))
    lse = np.zeros(N)
    for i0 in range(0, N, tile):
        qi = q[i0:i0 + tile]
        r = qi.shape[0]
        m = np.full(r, -np.inf)
        l = np.zeros(r)
        acc = np.zeros((r, d))
        for j0 in range(0, min(N, i0 + r), tile):
            s = scale * qi @ k[j0:j0 + tile].T
            rows = np.arange(i0, i0 + r)[:, None]
            cols = np.arange(j0, j0 + s.shape[1])[None, :]
            s = np.where(cols <= rows, s, -np.inf)
            m_new = np.maximum(m, s.max(1))
            p = np.exp(s - m_new[:, None])
            c = np.exp(m - m_new)
            l = c * l + p.sum(1)
            acc = c[:, None] * acc + p @ v[j0:j0 + tile]
            m = m_new
        o[i0:i0 + r] = acc / l[:, None]
        lse[i0:i0 + r] = m + np.log(l)
    return o, lse


def test_toy_run_tiled_prefill(golden):
    g = golden("toy_run.txt")
    N, d, tile = int(g["prefill_seqlen"]), int(g["prefill_head_dim"]), int(g["prefill_tile"])
    x = W.make_prefill(1, 1, 1, N, d, seed=0)
    q, k, v = _f64(x.q)[0, 0], _f64(x.k)[0, 0], _f64(x.v)[0, 0]
    ot, lt = _tiled_prefill_head(q, k, v, x.scale, tile)
    oo, lo = oracle.prefill(x.q, x.k, x.v, x.scale, True)
    # The page measured 1.1e-15; allow a little more for our own summation order.
    assert np.abs(ot - oo[0, 0]).max() <= 100 * g["prefill_max_abs_diff"]
    assert np.abs(lt - lo[0, 0]).max() <= TOL


def test_toy_run_split_decode(golden):
    g = golden("toy_run.txt")
    H, L, chunk = int(g["decode_query_heads"]), int(g["decode_cache_len"]), int(g["decode_chunk"])
    x = W.make_decode_contiguous(1, H, H, 128, L, seed=0)
    q = _f64(x.q)[0]
    kc, vc = _f64(x.k_cache)[0], _f64(x.v_cache)[0]
    o_parts, l_parts = [], []
    for t0 in range(0, L, chunk):              # each chunk: its own online softmax
        oh, lh = [], []
        for h in range(H):
            s = x.scale * kc[t0:t0 + chunk, h] @ q[h]
            _, o, lse = _online_blocks(s, vc[t0:t0 + chunk, h], 64)
            oh.append(o)
            lh.append(lse)
        o_parts.append(np.stack(oh))
        l_parts.append(np.array(lh))
    o_parts, l_parts = np.stack(o_parts), np.stack(l_parts)
    w = np.exp(l_parts - l_parts.max(0))       # merge by LSE weights (test-only)
    o_split = (w[..., None] * o_parts).sum(0) / w.sum(0)[..., None]
    oo, lo = oracle.decode(x.q, x.k_cache, x.v_cache, None, [L], x.scale)
    assert np.abs(o_split - oo[0]).max() <= 100 * g["decode_max_abs_diff"]


# ---------------------------------------------------------------------------
# Planted mistakes: every mutation must break at least one pin.
# ---------------------------------------------------------------------------

def _pins():
    return {"bruteforce": (_pin_bruteforce, TOL), "sdpa": (_pin_sdpa, 1e-12),
            "closed": (_pin_closed_forms, TOL), "gqa": (_pin_gqa, TOL),
            "combine": (_pin_combine, TOL), "partials": (_pin_partials_bruteforce, TOL),
            "append": (_pin_append, TOL),
            "varlen": (_pin_varlen, TOL), "variants": (_pin_variants, TOL),
            "varlen_variants": (_pin_varlen_variants, TOL)}


def _any_pin_fails():
    """Names of the pins whose error exceeds their tolerance.  A pin that
    raises is not a catch: the exception propagates and fails the test, so a
    planted mistake counts as caught only when some pin computes and
    disagrees."""
    failed = []
    for name, (fn, tol) in _pins().items():
        err = fn()
        if not (err <= tol):
            failed.append(name)
    return failed


def test_pins_pass_unmutated():
    assert _any_pin_fails() == []


@pytest.mark.parametrize("mutation", ["gqa_modulo", "strict_mask", "no_scale", "lse_no_max",
                                      "combine_unweighted", "gqa_off_by_one",
                                      "append_off_by_one", "append_not_attended",
                                      "varlen_cross_sequence", "window_off_by_one",
                                      "softcap_unscaled", "alibi_sign",
                                      "partials_softcap_dropped", "partials_alibi_dropped"])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    orig_ma = ref.masked_attention
    orig_comb = ref.combine
    if mutation == "gqa_modulo":
        monkeypatch.setattr(ref, "_kv_head", lambda h, nq, nkv: h % nkv)
    elif mutation == "gqa_off_by_one":
        monkeypatch.setattr(ref, "_kv_head", lambda h, nq, nkv: min(nkv - 1, (h + 1) // (nq // nkv)))
    elif mutation == "strict_mask":
        def strict(r0, r1, ncols):
            return np.arange(ncols)[None, :] < np.arange(r0, r1)[:, None]
        monkeypatch.setattr(ref, "_causal_allowed", strict)
    elif mutation == "no_scale":
        monkeypatch.setattr(ref, "masked_attention",
                            lambda q, k, v, scale, *a, **kw: orig_ma(q, k, v, 1.0, *a, **kw))
    elif mutation == "lse_no_max":
        def bad(q, k, v, scale, allowed=None, softcap=0.0, bias=None):
            o, lse = orig_ma(q, k, v, scale, allowed, softcap, bias)
            if len(k) and len(q):
                s = scale * (ref._f64(q) @ ref._f64(k).T)
                if softcap > 0:
                    s = softcap * np.tanh(s / softcap)
                if bias is not None:
                    s = s + bias
                if allowed is not None:
                    s = np.where(allowed, s, -np.inf)
                m = s.max(axis=1)
                lse = lse - np.where(np.isfinite(m), m, 0.0)   # dropped the max term
            return o, lse
        monkeypatch.setattr(ref, "masked_attention", bad)
    elif mutation == "window_off_by_one":
        orig_wa = ref._window_allowed
        monkeypatch.setattr(ref, "_window_allowed",
                            lambda r0, r1, n, c, w: orig_wa(r0, r1, n, c, w - 1 if w > 0 else w))
    elif mutation == "softcap_unscaled":
        def bad_cap(q, k, v, scale, allowed=None, softcap=0.0, bias=None):
            # cap * tanh(s) instead of cap * tanh(s / cap): the same as the
            # right formula applied to scores scaled by cap
            return orig_ma(q, k, v, scale * softcap if softcap > 0 else scale, allowed, softcap,
                           bias)
        monkeypatch.setattr(ref, "masked_attention", bad_cap)
    elif mutation == "alibi_sign":
        monkeypatch.setattr(ref, "_alibi", lambda slope, r, c: slope * np.abs(r[:, None] - c[None, :]))
    elif mutation == "varlen_cross_sequence":
        # sequences attend to the previous one's rows too (no per-example masking)
        monkeypatch.setattr(ref, "_seq_bounds", lambda cu: [(0, int(b)) for b in
                                                            np.asarray(cu).reshape(-1)[1:]])
    elif mutation == "append_off_by_one":
        monkeypatch.setattr(ref, "_append_position", lambda n: n + 1)
    elif mutation == "append_not_attended":
        orig_dec = ref.decode
        monkeypatch.setattr(ref, "decode", lambda q, kc, vc, bt, lens, scale, bs=0, **kw:
                            orig_dec(q, kc, vc, bt, [n - 1 for n in lens], scale, bs, **kw))
    elif mutation in ("partials_softcap_dropped", "partials_alibi_dropped"):
        # the per-split partials forget one variant (the whole-row decode keeps it)
        orig_part = ref.decode_partials
        drop = "softcap" if mutation == "partials_softcap_dropped" else "alibi_slopes"

        def bad_part(*a, **kw):
            kw.pop(drop, None)
            return orig_part(*a, **kw)
        monkeypatch.setattr(ref, "decode_partials", bad_part)
        monkeypatch.setattr(oracle, "decode_partials", bad_part)
    elif mutation == "combine_unweighted":
        monkeypatch.setattr(ref, "combine", lambda o, l: (ref._f64(o).mean(0), ref._f64(l).max(0)))
        monkeypatch.setattr(oracle, "combine", ref.combine)
    failed = _any_pin_fails()
    monkeypatch.setattr(ref, "masked_attention", orig_ma)
    monkeypatch.setattr(ref, "combine", orig_comb)
    assert failed, f"mutation {mutation} was not caught by any pin"


def test_sampled_rows_match_full_prefill():
    """The sampled-row entry point (used at sizes where every row is too slow)
    agrees with the pinned full prefill, causal and not, with GQA."""
    x = W.make_prefill(2, 6, 2, 90, 16, seed=9)
    rows = [(b, h, i) for b in range(2) for h in range(6) for i in (0, 1, 31, 64, 89)]
    for causal in (True, False):
        of, lf = oracle.prefill(x.q, x.k, x.v, x.scale, causal)
        orow, lrow = oracle.prefill_rows(x.q, x.k, x.v, x.scale, causal, rows)
        for n, (b, h, i) in enumerate(rows):
            assert np.abs(orow[n] - of[b, h, i]).max() <= TOL
            assert abs(lrow[n] - lf[b, h, i]) <= TOL
