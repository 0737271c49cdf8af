"""Seeded synthetic inputs for causal GQA partial attention with logical CP shards.

This module is shared by the tests, the bench and the smoke check.  It only draws
random numbers and lays them out in the buffers that both the oracle and the CUDA
path consume; it computes none of the attention, partition, interleave or merge
arithmetic.  Every tensor is drawn on the CPU with a seeded ``torch.Generator`` so
that the oracle and the GPU see identical bits (bf16 values are exactly
representable in float64).

Workloads (shapes follow the synthetic stand-ins for the pages' serving workload,
a Qwen2.5-3B gsm8k run whose data and weights are not used):

* ``tiny``    1 x 256 tokens, 4 q heads / 1 kv head, d=64, fp32, cp=2, pass-KV.
* ``full``    1 x 8192 tokens, 16/2 heads, d=128, bf16, cp=2, pass-KV.
* ``long``    2 x 32768 tokens, 16/2 heads, d=128, bf16, cp=4, pass-KV.
* ``chunked`` 4 seqs x (2048 new queries over 32768 cached+new kv), 16/2 heads,
  d=128, bf16, paged kv (block 16), cp=4, interleave 8, pass-Q.
* ``decode``  64 seqs, one query each, context ~ U[1024, 32768], 32/8 heads,
  d=128, bf16, paged kv (block 16), cp=2, interleave 8.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "Workload", "WORKLOADS", "prefill_inputs", "paged_inputs", "decode_lengths",
    "normal", "shuffled_block_tables", "block_capacity",
]


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "pass_kv" | "pass_q" | "decode"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: torch.dtype
    cp: int
    seq_len: int = 0          # pass_kv: tokens per sequence
    q_len: int = 0            # pass_q: new query tokens per sequence
    kv_len: int = 0           # pass_q: cached + new kv tokens per sequence
    min_len: int = 0          # decode: context length range (inclusive)
    max_len: int = 0
    interleave: int = 8
    block_size: int = 16
    seed: int = 0             # values
    table_seed: int = 0       # block-table shuffles
    len_seed: int = 0         # decode lengths
    sample_rows: int = 0      # rows per (seq, head) the oracle checks at full size; 0 = all
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", "pass_kv", 1, 4, 1, 64, torch.float32, 2, seq_len=256, seed=1000),
    "full": Workload("full", "pass_kv", 1, 16, 2, 128, torch.bfloat16, 2, seq_len=8192, seed=1001),
    "long": Workload("long", "pass_kv", 2, 16, 2, 128, torch.bfloat16, 4, seq_len=32768,
                     seed=1002, sample_rows=512),
    "chunked": Workload("chunked", "pass_q", 4, 16, 2, 128, torch.bfloat16, 4, q_len=2048,
                        kv_len=32768, interleave=8, block_size=16, seed=1003, table_seed=2003,
                        sample_rows=512),
    "decode": Workload("decode", "decode", 64, 32, 8, 128, torch.bfloat16, 2, min_len=1024,
                       max_len=32768, interleave=8, block_size=16, seed=1004, table_seed=2004,
                       len_seed=3000),
}


def normal(shape, dtype, gen: torch.Generator) -> torch.Tensor:
    """N(0, 1) values drawn in fp32 and rounded to ``dtype`` (CPU)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def prefill_inputs(seq_lens, num_q_heads, num_kv_heads, head_dim, dtype, seed):
    """Token-major varlen Q/K/V for pass-KV prefill.

    Returns a dict with ``q`` [sum T, Hq, d], ``k``/``v`` [sum T, Hkv, d] and
    ``cu_seqlens`` int32 [B + 1] (all CPU tensors).
    """
    g = torch.Generator().manual_seed(seed)
    total = int(sum(seq_lens))
    q = normal((total, num_q_heads, head_dim), dtype, g)
    k = normal((total, num_kv_heads, head_dim), dtype, g)
    v = normal((total, num_kv_heads, head_dim), dtype, g)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    return {"q": q, "k": k, "v": v, "cu_seqlens": cu}


def block_capacity(kv_len: int, cp: int, interleave: int, block_size: int) -> int:
    """Pages reserved per (rank, sequence).

    Allocation policy only: room for ceil(kv_len / cp) + interleave tokens, which
    is never less than what any rank receives from a round-robin deal of groups of
    ``interleave`` tokens.
    """
    room = -(-kv_len // cp) + interleave
    return -(-room // block_size)


def shuffled_block_tables(capacities, cp, gen: torch.Generator):
    """Per-rank block tables over per-rank page pools.

    Rank r owns a pool of ``sum(capacities)`` pages; its table row for sequence b
    lists ``capacities[b]`` distinct pool ids drawn from a seeded permutation, and
    is padded with -1 up to ``max(capacities)`` entries.

    Returns (block_tables int32 [cp, B, max_blocks], pool_pages).
    """
    B = len(capacities)
    max_blocks = max(capacities) if B else 0
    pool = int(sum(capacities))
    tables = torch.full((cp, B, max_blocks), -1, dtype=torch.int32)
    for r in range(cp):
        perm = torch.randperm(pool, generator=gen).to(torch.int32)
        off = 0
        for b, c in enumerate(capacities):
            tables[r, b, :c] = perm[off:off + c]
            off += c
    return tables, pool


def paged_inputs(num_seqs, q_len, kv_lens, num_q_heads, num_kv_heads, head_dim, dtype, cp,
                 interleave, block_size, seed, table_seed, q_is_decode=False):
    """Paged, per-rank KV pools plus queries (pass-Q chunked prefill or decode).

    * ``k_cache``/``v_cache``: [cp, pool_pages, Hkv, block_size, d] -- one pool per
      logical rank, head-major pages, every slot filled with N(0, 1).
    * ``block_tables``: int32 [cp, B, max_blocks] (seeded shuffle, -1 padding).
    * ``seq_lens``: int32 [B] kv lengths (cached + new).
    * ``q``: decode: [B, Hq, d]; chunked prefill: [B * q_len, Hq, d] with
      ``cu_seqlens_q`` int32 [B + 1].
    """
    g = torch.Generator().manual_seed(seed)
    gt = torch.Generator().manual_seed(table_seed)
    caps = [block_capacity(int(L), cp, interleave, block_size) for L in kv_lens]
    tables, pool = shuffled_block_tables(caps, cp, gt)
    if q_is_decode:
        q = normal((num_seqs, num_q_heads, head_dim), dtype, g)
        cu_q = torch.arange(num_seqs + 1, dtype=torch.int32)
    else:
        q = normal((num_seqs * q_len, num_q_heads, head_dim), dtype, g)
        cu_q = torch.arange(num_seqs + 1, dtype=torch.int32) * q_len
    shape = (cp, pool, num_kv_heads, block_size, head_dim)
    k_cache = normal(shape, dtype, g)
    v_cache = normal(shape, dtype, g)
    return {
        "q": q, "k_cache": k_cache, "v_cache": v_cache, "block_tables": tables,
        "seq_lens": torch.tensor([int(L) for L in kv_lens], dtype=torch.int32),
        "cu_seqlens_q": cu_q,
    }


def decode_lengths(num_seqs, min_len, max_len, seed):
    """Context lengths ~ U{min_len..max_len} (int32 [B], seeded)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(min_len, max_len + 1, (num_seqs,), generator=g, dtype=torch.int64).to(
        torch.int32)


def workload_inputs(w: Workload):
    """All inputs of a named workload at its full size (CPU tensors)."""
    if w.kind == "pass_kv":
        return prefill_inputs([w.seq_len] * w.num_seqs, w.num_q_heads, w.num_kv_heads,
                              w.head_dim, w.dtype, w.seed)
    if w.kind == "pass_q":
        return paged_inputs(w.num_seqs, w.q_len, [w.kv_len] * w.num_seqs, w.num_q_heads,
                            w.num_kv_heads, w.head_dim, w.dtype, w.cp, w.interleave,
                            w.block_size, w.seed, w.table_seed)
    if w.kind == "decode":
        lens = decode_lengths(w.num_seqs, w.min_len, w.max_len, w.len_seed).tolist()
        return paged_inputs(w.num_seqs, 1, lens, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.dtype, w.cp, w.interleave, w.block_size, w.seed, w.table_seed,
                            q_is_decode=True)
    raise ValueError(w.kind)


def sample_rows(n_rows: int, chunk_starts, count: int, seed: int):
    """Seeded, stratified subset of query rows of one sequence (sorted, unique).

    Always holds row 0, the last row and the first and last row of every chunk
    (``chunk_starts`` lists chunk start rows, with the end as last entry); the rest is
    spread over the chunks in proportion to their size.
    """
    if count >= n_rows:
        return list(range(n_rows))
    g = torch.Generator().manual_seed(seed)
    keep = {0, n_rows - 1}
    for a, b in zip(chunk_starts[:-1], chunk_starts[1:]):
        if b > a:
            keep.update((a, b - 1))
    remaining = max(count - len(keep), 0)
    nchunks = max(len(chunk_starts) - 1, 1)
    per = int(math.ceil(remaining / nchunks))
    for a, b in zip(chunk_starts[:-1], chunk_starts[1:]):
        if b > a and per > 0:
            idx = torch.randint(a, b, (per,), generator=g).tolist()
            keep.update(idx)
    return sorted(keep)
