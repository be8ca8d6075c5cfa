"""Shared helpers for the GPU parity tests (tolerances and comparisons)."""

import numpy as np
import torch

# Acceptance bar for bf16 inputs with fp32 accumulation against the float64
# oracle: O max-abs 2e-2 and mean-abs 2e-3, LSE max-abs 1e-3.
O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def nan_like(shape, device):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=device)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", lse_rel=0.0):
    """Element-wise parity: returns (max|dO|, mean|dO|, max|dLSE|).

    lse_rel adds a tolerance proportional to |LSE| for values whose fp32
    representation itself is coarser than LSE_MAX (ALiBi partials far from
    the query reach |LSE| ~ 1e4, where one fp32 step is ~1e-3)."""
    o = o_gpu.detach().double().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else o_gpu
    lse = lse_gpu.detach().double().cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output (unwritten element?)"
    # -inf LSE (empty key set) must match exactly; finite ones within tolerance.
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), inf_ref), f"{what}: -inf pattern of LSE differs"
    assert np.isfinite(lse[~inf_ref]).all(), f"{what}: non-finite LSE"
    err = np.abs(o - o_ref)
    fin = ~inf_ref
    lerr = (np.abs(lse[fin] - lse_ref[fin]) - lse_rel * np.abs(lse_ref[fin])).max() if fin.any() else 0.0
    emax, emean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert emax <= O_MAX and emean <= O_MEAN and lerr <= LSE_MAX, \
        f"{what}: max|dO|={emax:.3e} mean|dO|={emean:.3e} max|dLSE|={lerr:.3e}"
    return emax, emean, float(lerr)


def split_ranges(kv_len: int, num_splits: int, window_left: int = -1):
    """Tokens attended by every split under the split rule the C header states
    for attn_decode_splitkv(_ex), restated here for the tests:
    c = roundup(ceil(len / S), 16); split s covers [s*c, min((s+1)*c, len)).
    With a sliding window the rule applies from lo16 (the window's first
    token lo rounded down to a multiple of 16) and tokens below lo are dropped."""
    lo = max(0, kv_len - 1 - window_left) if window_left >= 0 else 0
    lo16 = lo // 16 * 16
    n = kv_len - lo16
    per = -(-n // num_splits)
    c = -(-per // 16) * 16
    out = []
    for s in range(num_splits):
        a, b = lo16 + min(s * c, n), lo16 + min(min(s * c, n) + c, n)
        out.append((min(max(a, lo), b), b))
    return out
