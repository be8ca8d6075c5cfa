"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, and it imports neither the CUDA binding nor the oracle.

Recipe (one CPU ``torch.Generator`` per workload, seeded, draws in a fixed
order): values are ``torch.randn`` float32 rounded to bfloat16 (round to
nearest even).  The shapes follow the attention layers the pages measure:
Qwen2.5-7B (28 query / 4 key-value heads, head_dim 128) and Llama-3-8B
(32 / 8, head_dim 128), from "The Inference Wall, Part 8" and "FlashAttention
for inference: tiled prefill and split-KV decoding".
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

BF16 = torch.bfloat16


@dataclass
class PrefillInputs:
    q: torch.Tensor          # (B, n_q, N, d) bf16
    k: torch.Tensor          # (B, n_kv, N, d) bf16
    v: torch.Tensor          # (B, n_kv, N, d) bf16
    scale: float
    causal: bool = True

    @property
    def shape(self):
        B, n_q, N, d = self.q.shape
        return B, n_q, self.k.shape[1], N, d


@dataclass
class DecodeInputs:
    q: torch.Tensor                      # (B, n_q, d) bf16
    k_cache: torch.Tensor                # paged (nb, bs, n_kv, d) or contiguous (B, L, n_kv, d)
    v_cache: torch.Tensor
    block_table: Optional[torch.Tensor]  # (B, max_blocks) int32, or None (contiguous)
    kv_lens: torch.Tensor                # (B,) int32
    block_size: int                      # tokens per block; 0 for a contiguous cache
    scale: float
    max_kv_len: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def n_kv(self) -> int:
        return self.k_cache.shape[2]


def _randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(BF16)


def make_prefill(batch: int, n_q: int, n_kv: int, seqlen: int, head_dim: int,
                 seed: int = 0, spike_frac: float = 0.0, spike_scale: float = 8.0,
                 causal: bool = True) -> PrefillInputs:
    """Q, K, V iid N(0,1) in bf16, drawn in the order Q, K, V.

    With ``spike_frac`` > 0, for each (sequence, kv head) floor(spike_frac*N)
    key positions, drawn without replacement after V, are multiplied by
    ``spike_scale`` (8 is a power of two, so the product is exact in bf16).
    This makes a row's running maximum jump part-way through the keys.
    """
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (batch, n_q, seqlen, head_dim))
    k = _randn_bf16(gen, (batch, n_kv, seqlen, head_dim))
    v = _randn_bf16(gen, (batch, n_kv, seqlen, head_dim))
    n_spike = int(math.floor(spike_frac * seqlen))
    if n_spike > 0:
        for b in range(batch):
            for h in range(n_kv):
                pos = torch.randperm(seqlen, generator=gen)[:n_spike]
                k[b, h, pos] = (k[b, h, pos].float() * spike_scale).to(BF16)
    return PrefillInputs(q, k, v, 1.0 / math.sqrt(head_dim), causal)


def make_decode_contiguous(batch: int, n_q: int, n_kv: int, head_dim: int,
                           kv_len: int, seed: int = 0,
                           max_kv_len: Optional[int] = None) -> DecodeInputs:
    """Contiguous cache (B, max_kv_len, n_kv, d); every sequence holds kv_len
    tokens.  Draw order: q, K cache, V cache."""
    L = kv_len if max_kv_len is None else max_kv_len
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (batch, n_q, head_dim))
    k = _randn_bf16(gen, (batch, L, n_kv, head_dim))
    v = _randn_bf16(gen, (batch, L, n_kv, head_dim))
    lens = torch.full((batch,), kv_len, dtype=torch.int32)
    return DecodeInputs(q, k, v, None, lens, 0, 1.0 / math.sqrt(head_dim), L)


def make_decode_paged(batch: int, n_q: int, n_kv: int, head_dim: int,
                      kv_lens, block_size: int = 16, seed: int = 0,
                      extra_blocks: int = 0) -> DecodeInputs:
    """Paged cache (num_blocks, block_size, n_kv, d) with a block table.

    Physical blocks = sum ceil(len / block_size) (+ ``extra_blocks`` unused
    ones); they are assigned to (sequence, logical block) by a seeded random
    permutation.  Unused block-table entries are 0 and are never read.  Draw
    order: q, K cache, V cache, permutation.
    """
    gen = torch.Generator().manual_seed(seed)
    lens = torch.as_tensor(list(kv_lens), dtype=torch.int32)
    assert lens.numel() == batch
    nblk = [(int(n) + block_size - 1) // block_size for n in lens.tolist()]
    total = sum(nblk) + extra_blocks
    max_blocks = max(1, max(nblk) if nblk else 1)
    q = _randn_bf16(gen, (batch, n_q, head_dim))
    k = _randn_bf16(gen, (max(total, 1), block_size, n_kv, head_dim))
    v = _randn_bf16(gen, (max(total, 1), block_size, n_kv, head_dim))
    perm = torch.randperm(max(total, 1), generator=gen)
    table = torch.zeros((batch, max_blocks), dtype=torch.int32)
    pos = 0
    for b in range(batch):
        for j in range(nblk[b]):
            table[b, j] = int(perm[pos])
            pos += 1
    max_len = int(lens.max()) if batch else 0
    return DecodeInputs(q, k, v, table, lens, block_size,
                        1.0 / math.sqrt(head_dim), max_len)


@dataclass
class VarlenInputs:
    q: torch.Tensor            # (n_q, total, d) bf16, sequences packed end to end
    k: torch.Tensor            # (n_kv, total, d) bf16
    v: torch.Tensor
    cu_seqlens: torch.Tensor   # (num_seqs + 1,) int32
    scale: float
    causal: bool = True


def make_prefill_varlen(lens, n_q: int, n_kv: int, head_dim: int, seed: int = 0,
                        extra_rows: int = 0, causal: bool = True) -> VarlenInputs:
    """Sequences of the given lengths packed end to end (head-major), plus
    ``extra_rows`` rows that belong to no sequence.  Draw order: Q, K, V."""
    lens = [int(n) for n in lens]
    T = sum(lens) + extra_rows
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (n_q, T, head_dim))
    k = _randn_bf16(gen, (n_kv, T, head_dim))
    v = _randn_bf16(gen, (n_kv, T, head_dim))
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.as_tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return VarlenInputs(q, k, v, cu, 1.0 / math.sqrt(head_dim), causal)


def paged_lens_uniform(batch: int, lo: int, hi: int, seed: int = 0):
    """Integer-uniform sequence lengths in [lo, hi] inclusive (seeded)."""
    gen = torch.Generator().manual_seed(seed + 1)
    return torch.randint(lo, hi + 1, (batch,), generator=gen, dtype=torch.int64).tolist()


# ---------------------------------------------------------------------------
# The five workloads of the hot path (sizes only; see the design notes).
# ---------------------------------------------------------------------------

def tiny_prefill(seed: int = 0) -> PrefillInputs:
    """Causal prefill, batch 1, 1 head, N=256, head_dim 64."""
    return make_prefill(1, 1, 1, 256, 64, seed=seed)


def qwen_prefill(seqlen: int = 8192, seed: int = 0) -> PrefillInputs:
    """Qwen2.5-7B attention layer: 28 query / 4 kv heads, head_dim 128."""
    return make_prefill(1, 28, 4, seqlen, 128, seed=seed)


def llama_long_prefill(seqlen: int = 32768, seed: int = 0) -> PrefillInputs:
    """Llama-3-8B attention layer at long context, 1% of keys scaled by 8."""
    return make_prefill(1, 32, 8, seqlen, 128, seed=seed, spike_frac=0.01)


def qwen_decode(kv_len: int = 30720, seed: int = 0) -> DecodeInputs:
    """Single-token decode, 28 / 4 heads, head_dim 128, contiguous cache."""
    return make_decode_contiguous(1, 28, 4, 128, kv_len, seed=seed)


def qwen_varlen_prefill(seed: int = 0, num_seqs: int = 16, lo: int = 256,
                        hi: int = 4096) -> VarlenInputs:
    """A prefill batch of prompts of different lengths (integer-uniform in
    [lo, hi], seeded) packed without padding, 28 / 4 heads, head_dim 128."""
    lens = paged_lens_uniform(num_seqs, lo, hi, seed + 7)
    return make_prefill_varlen(lens, 28, 4, 128, seed=seed)


def llama_paged_decode(seed: int = 0, batch: int = 16) -> DecodeInputs:
    """16 sequences, lengths uniform in [1024, 32768], 32 / 8 heads,
    head_dim 128, 16-token blocks."""
    lens = paged_lens_uniform(batch, 1024, 32768, seed)
    return make_decode_paged(batch, 32, 8, 128, lens, block_size=16, seed=seed)
