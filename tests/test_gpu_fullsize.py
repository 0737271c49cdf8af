"""Parity at the workloads' full sizes, in the launch configurations bench.py times (partials +
merge, and the fused launches).

The oracle computes sampled query rows one by one (stratified: every chunk, its first and last
rows, row 0 and the last row, 512 rows per sequence); decode is checked on every row.
"""
import math

import numpy as np
import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_merged, check_partials

pytestmark = pytest.mark.gpu


def _rows(w, T, cu_start, seed):
    bnd = orc.chunk_bounds(T, w.cp).tolist()
    return [cu_start + r for r in wl.sample_rows(T, bnd, w.sample_rows or 512, seed)]


@pytest.mark.parametrize("name", ["full", "long"])
def test_pass_kv_full_size(lib, name):
    w = wl.WORKLOADS[name]
    x = wl.workload_inputs(w)
    q, k, v, cu = (x[n].cuda() for n in ("q", "k", "v", "cu_seqlens"))
    out, lse = lib.cp_partial_attn_prefill(q, cu, w.cp, k=k, v=v, max_seqlen_q=w.seq_len)
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=w.dtype)
    rows = []
    for b in range(w.num_seqs):
        rows += _rows(w, w.seq_len, b * w.seq_len, 40 + b)
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], w.cp,
                                1 / math.sqrt(w.head_dim), rows=rows)
    check_partials(out, lse, O, L, rows=rows, what=f"{name} partials")
    Om, Lm = orc.lse_merge(O, L)
    idx = torch.as_tensor(rows, device="cuda")
    check_merged(mo.index_select(0, idx), ml.index_select(0, idx), Om, Lm, what=f"{name} merged")
    fo, fl = lib.cp_attn_prefill_fused(q, cu, w.cp, k, v, max_seqlen_q=w.seq_len)
    check_merged(fo.index_select(0, idx), fl.index_select(0, idx), Om, Lm, what=f"{name} fused")


def test_pass_q_chunked_full_size(lib):
    w = wl.WORKLOADS["chunked"]
    x = wl.workload_inputs(w)
    dev = {n: x[n].cuda() for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens", "cu_seqlens_q")}
    out, lse = lib.cp_partial_attn_prefill(
        dev["q"], dev["cu_seqlens_q"], w.cp, mode=lib.CP_PASS_Q, k_cache=dev["k_cache"],
        v_cache=dev["v_cache"], block_tables=dev["block_tables"], seq_lens_kv=dev["seq_lens"],
        interleave=w.interleave, max_seqlen_q=w.q_len)
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=w.dtype)
    rows = []
    for b in range(w.num_seqs):
        rows += _rows(w, w.q_len, b * w.q_len, 60 + b)
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], w.cp, w.interleave, w.block_size,
                               1 / math.sqrt(w.head_dim), rows=rows)
    check_partials(out, lse, O, L, rows=rows, what="chunked partials")
    Om, Lm = orc.lse_merge(O, L)
    idx = torch.as_tensor(rows, device="cuda")
    check_merged(mo.index_select(0, idx), ml.index_select(0, idx), Om, Lm, what="chunked merged")
    fo, fl = lib.cp_attn_prefill_fused(
        dev["q"], dev["cu_seqlens_q"], w.cp, mode=lib.CP_PASS_Q, k_cache=dev["k_cache"],
        v_cache=dev["v_cache"], block_tables=dev["block_tables"], seq_lens_kv=dev["seq_lens"],
        interleave=w.interleave, max_seqlen_q=w.q_len)
    check_merged(fo.index_select(0, idx), fl.index_select(0, idx), Om, Lm, what="chunked fused")


def test_decode_full_size(lib):
    w = wl.WORKLOADS["decode"]
    x = wl.workload_inputs(w)
    lens = x["seq_lens"].tolist()
    dev = {n: x[n].cuda() for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    ns, st = lib.cp_decode_plan(w.num_seqs, w.num_kv_heads, w.cp, w.interleave, w.block_size,
                                max(lens))
    out, lse = lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"],
                                          dev["block_tables"], dev["seq_lens"], w.cp, w.interleave,
                                          num_splits=ns, split_tokens=st)
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=w.dtype)
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], w.cp, w.interleave, w.block_size,
                               1 / math.sqrt(w.head_dim))
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what="decode merged")
    fo, fl = lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                     dev["seq_lens"], w.cp, w.interleave, num_splits=ns,
                                     split_tokens=st)
    check_merged(fo, fl, Om, Lm, what="fused decode")


def test_pass_kv_single_128k_sequence(lib):
    """One sequence of 131072 tokens at cp = 8 (16 chunks of 8192 tokens, ~32K work items,
    8.6 GB of f32 partials): index arithmetic at the large end, checked on 256 stratified rows."""
    T, cp, Hq, Hkv, d = 131072, 8, 16, 2, 128
    x = wl.prefill_inputs([T], Hq, Hkv, d, torch.bfloat16, seed=660)
    q, k, v, cu = (x[n].cuda() for n in ("q", "k", "v", "cu_seqlens"))
    out, lse = lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=T)
    bnd = orc.chunk_bounds(T, cp).tolist()
    rows = wl.sample_rows(T, bnd, 256, 661)
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d),
                                rows=rows)
    check_partials(out, lse, O, L, rows=rows, what="128K partials")
    Om, Lm = orc.lse_merge(O, L)
    idx = torch.as_tensor(rows, device="cuda")
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=torch.bfloat16)
    check_merged(mo.index_select(0, idx), ml.index_select(0, idx), Om, Lm, what="128K merged")
    del out, lse, mo, ml
    fo, fl = lib.cp_attn_prefill_fused(q, cu, cp, k, v, max_seqlen_q=T)
    check_merged(fo.index_select(0, idx), fl.index_select(0, idx), Om, Lm, what="128K fused")
