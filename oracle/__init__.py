"""Float64 CPU oracle for causal GQA partial attention over logical CP shards.

TEST INFRASTRUCTURE, not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
``--impl reference`` arm) may import or run anything under ``oracle/``.  The CUDA
path never calls it and it never calls the CUDA path; the two share no code.

Sources (vLLM pull-request pages):
  * "Add utility functions to enable pass-kv prefill and allgather decode"
    (PR 26059), Purpose -- attention is the only op that couples tokens; prefill
    shards Q and KV and exchanges Q or KV shards around partial attention; decode
    keeps KV round-robin over the CP ranks; partial attention (MLSys paper linked
    there) is merged afterwards.
  * "[Feature] Prefill Context Parallel (PCP) basic support" (PR 28718), Purpose
    and code-review summary -- block tables extended for DCP/PCP; the kv-cache
    interleave size applies to both prefill and decode CP.
  * "[Feature] Support Prefill Context Parallel (PCP) for GQA flashinfer"
    (PR 28723), Test Plan -- interleave size 8, GQA model.

Every function here is pinned by ``tests/test_oracle_*.py`` (brute force, a
library routine, closed forms, invariants).  Parity unpinned: none of the
functions; the *choice* of placing chunked-prefill KV by the round-robin deal is a
reading of the pages (both readings give the same attention output).
"""
from .cp_oracle import (  # noqa: F401
    chunk_bounds, shard_chunks, partition, interleave_deal, local_lengths, rank_positions,
    slot_mapping, partial_attention, attention, lse_merge, pass_kv_partials, pass_q_partials,
    decode_partials, gather_rank_kv, kv_cache_write,
)
