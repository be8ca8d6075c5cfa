"""The allocation-free decode entry point, attn_decode_noalloc.

Callers that cannot allocate device memory on their decode path (a serving
loop that reserved all memory at start-up, a plugin whose host framework owns
the allocator, a step that must not pay cudaMalloc's synchronisation) use this
call: it keeps the split partials in the library's fixed device buffer instead
of caller-provided ones.  These tests call it through the C ABI and check that
two calls in a row give the same results, within the usual tolerance, as the
allocating entry points attn_decode_splitkv + attn_combine with the same split
count; and that a request larger than the buffer is refused before any launch.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""

import pytest
import torch

import exact_io_aware_order_gb300 as attn
from exact_io_aware_order_gb300 import workloads as W
from exact_io_aware_order_gb300._lib import ATTN_NOALLOC_SCRATCH_BYTES, lib, status_codes
from gpu_util import O_MAX, LSE_MAX, nan_like

pytestmark = pytest.mark.gpu


def _noalloc(d, dev, S, o, lse):
    """One call of attn_decode_noalloc through ctypes on the current stream."""
    bt = d.block_table
    paged = bt is not None
    B, Hq, D = d.q.shape
    st = lib().attn_decode_noalloc(
        d._q.data_ptr(), d._k.data_ptr(), d._v.data_ptr(), d._bt.data_ptr() if paged else None,
        d._lens.data_ptr(), S, o.data_ptr(), lse.data_ptr(), B, Hq, d.n_kv, D,
        d.block_size if paged else 0, bt.shape[1] if paged else 0,
        d.k_cache.shape[0] if paged else 0, d.max_kv_len, d.scale,
        torch.cuda.current_stream().cuda_stream)
    return st


def _to_dev(d, dev):
    d._q, d._k, d._v = d.q.to(dev), d.k_cache.to(dev), d.v_cache.to(dev)
    d._lens = d.kv_lens.to(dev)
    d._bt = d.block_table.to(dev) if d.block_table is not None else None
    return d


@pytest.mark.parametrize("case", ["qwen_auto", "qwen_16", "paged_4", "paged_empty_seq",
                                  "d256"])
def test_noalloc_matches_allocating_entry_points(dev, case):
    if case.startswith("qwen"):
        d = W.qwen_decode(30720)
        S = 0 if case == "qwen_auto" else 16
    elif case == "paged_4":
        d = W.llama_paged_decode()
        S = 4
    elif case == "d256":
        d = W.make_decode_paged(2, 16, 8, 256, [5000, 17], block_size=16, seed=7)
        S = 0
    else:
        d = W.make_decode_paged(3, 8, 2, 128, [0, 700, 33], block_size=16, seed=5)
        S = 3
    _to_dev(d, dev)
    # The existing, allocating entry points with the same split count.
    S_eff = S if S else attn.decode_num_splits(d.q.shape[0], d.n_kv, d.max_kv_len)
    op, lp = attn.decode_splitkv(d._q, d._k, d._v, d._lens, d._bt, num_splits=S_eff,
                                 max_kv_len=d.max_kv_len, scale=d.scale)
    o_ref, l_ref = attn.combine(op, lp)
    attn.check_device_status()
    B, Hq, D = d.q.shape
    for call in range(2):  # two calls in a row share (and overwrite) the buffer
        o, lse = nan_like((B, Hq, D), dev), nan_like((B, Hq), dev)
        assert _noalloc(d, dev, S, o, lse) == 0
        attn.check_device_status()
        assert torch.isfinite(o).all()
        assert (o - o_ref).abs().max().item() <= O_MAX
        fin = torch.isfinite(l_ref)
        assert torch.equal(torch.isneginf(lse), torch.isneginf(l_ref))
        if fin.any():
            assert (lse[fin] - l_ref[fin]).abs().max().item() <= LSE_MAX


def test_noalloc_refuses_requests_beyond_its_buffer(dev):
    d = _to_dev(W.make_decode_contiguous(16, 32, 8, 128, 64, seed=1), dev)
    S = 1024  # 1024 * 16 * 32 * 129 * 4 bytes is far above the buffer
    assert S * 16 * 32 * 129 * 4 > ATTN_NOALLOC_SCRATCH_BYTES
    o, lse = nan_like((16, 32, 128), dev), nan_like((16, 32), dev)
    assert _noalloc(d, dev, S, o, lse) == status_codes()["ATTN_ERR_SCRATCH"]
    torch.cuda.synchronize()
    assert torch.isnan(o).all()  # nothing was launched
