"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each one.

A pin set that lets a dropped term, a wrong sign or index, or a swapped operand through
would not be worth trusting; every mutation below must make at least one pin fail.
"""
import math

import numpy as np
import pytest

from oracle import cp_oracle as orc
import tests.test_oracle_pins as pins

_orig_pa = orc.partial_attention
_orig_merge = orc.lse_merge
_orig_gather = orc.gather_rank_kv


def _strict_causal(q, k, v, q_pos, k_pos, scale, **kw):
    return _orig_pa(q, k, v, q_pos, np.asarray(k_pos) + 1, scale, **kw)


def _wrong_gqa(q, k, v, q_pos, k_pos, scale, **kw):
    k = np.roll(np.asarray(k, dtype=np.float64), 1, axis=1)
    v = np.roll(np.asarray(v, dtype=np.float64), 1, axis=1)
    return _orig_pa(q, k, v, q_pos, k_pos, scale, **kw)


def _swapped_kv(q, k, v, q_pos, k_pos, scale, **kw):
    return _orig_pa(q, v, k, q_pos, k_pos, scale, **kw)


def _negated_scale(q, k, v, q_pos, k_pos, scale, **kw):
    return _orig_pa(q, k, v, q_pos, k_pos, -scale, **kw)


def _lse_log2(q, k, v, q_pos, k_pos, scale, **kw):
    O, L = _orig_pa(q, k, v, q_pos, k_pos, scale, **kw)
    return O, L / math.log(2.0)


def _lse_bias(q, k, v, q_pos, k_pos, scale, **kw):
    O, L = _orig_pa(q, k, v, q_pos, k_pos, scale, **kw)
    return O, L + 1e-6


def _merge_plain_mean(O, L):
    O = np.asarray(O, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    fin = np.isfinite(L)
    n = np.maximum(fin.sum(axis=0), 1)
    Om = np.where(fin[..., None], np.nan_to_num(O), 0).sum(axis=0) / n[..., None]
    return Om, L.max(axis=0)


def _merge_unnormalised(O, L):
    Om, Lm = _orig_merge(O, L)
    L = np.asarray(L, dtype=np.float64)
    M = L.max(axis=0)
    with np.errstate(invalid="ignore"):
        wsum = np.exp(Lm - M)
    return np.where(np.isfinite(Lm)[..., None], Om * wsum[..., None], 0.0), Lm


def _gather_reversed_pages(cache_r, table_row, n_local, block_size):
    row = np.asarray(table_row).copy()
    n_pages = -(-n_local // block_size)
    row[:n_pages] = row[:n_pages][::-1]
    return _orig_gather(cache_r, row, n_local, block_size)


def _chunk_bounds_ceil(T, cp):
    return np.array([-(-(k * T) // (2 * cp)) for k in range(2 * cp + 1)], dtype=np.int64)


def _shard_chunks_contiguous(r, cp):
    return (2 * r, 2 * r + 1)


def _deal_wrong_local(L, cp, I):
    p = np.arange(L, dtype=np.int64)
    rank = (p // I) % cp
    local = (p // (I * cp)) * I + (p % I) + (rank > 0)
    return rank, local


def _deal_wrong_rank(L, cp, I):
    p = np.arange(L, dtype=np.int64)
    rank = p % cp
    local = p // cp
    return rank, local


def _pass_kv_mutant(drop_ctx=False, bounds_over_q=False):
    """pass_kv_partials with one planted mistake in its cached-context handling."""
    def fn(q, k, v, cu_seqlens, cp, scale, rows=None, cu_seqlens_kv=None):
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        cu_kv = cu if cu_seqlens_kv is None else np.asarray(cu_seqlens_kv, dtype=np.int64)
        per_seq = orc._rows_by_seq(cu, rows)
        R = sum(x.size for x in per_seq)
        O = np.zeros((cp, R, q.shape[1], q.shape[2]))
        L = np.full((cp, R, q.shape[1]), -np.inf)
        out_row = 0
        for b in range(cu.size - 1):
            lo, hi, klo, khi = int(cu[b]), int(cu[b + 1]), int(cu_kv[b]), int(cu_kv[b + 1])
            ctx = 0 if drop_ctx else (khi - klo) - (hi - lo)
            sel = per_seq[b]
            bnd = orc.chunk_bounds((hi - lo) if bounds_over_q else (khi - klo), cp)
            for s_ in range(cp):
                keys = np.concatenate([np.arange(bnd[c], bnd[c + 1]) for c in orc.shard_chunks(s_, cp)])
                o, l = orc.partial_attention(q[lo:hi][sel], k[klo:khi][keys], v[klo:khi][keys],
                                             ctx + sel, keys, scale)
                O[s_, out_row:out_row + sel.size] = o
                L[s_, out_row:out_row + sel.size] = l
            out_row += sel.size
        return O, L
    return fn


MUTATIONS = {
    "pass_kv_ctx_dropped": ("pass_kv_partials", _pass_kv_mutant(drop_ctx=True)),
    "pass_kv_bounds_over_q_len": ("pass_kv_partials", _pass_kv_mutant(bounds_over_q=True)),
    "causal_strict": ("partial_attention", _strict_causal),
    "gqa_wrong_group": ("partial_attention", _wrong_gqa),
    "k_v_swapped": ("partial_attention", _swapped_kv),
    "scale_sign": ("partial_attention", _negated_scale),
    "lse_in_log2": ("partial_attention", _lse_log2),
    "lse_small_bias": ("partial_attention", _lse_bias),
    "merge_plain_mean": ("lse_merge", _merge_plain_mean),
    "merge_unnormalised": ("lse_merge", _merge_unnormalised),
    "gather_page_order": ("gather_rank_kv", _gather_reversed_pages),
    "chunk_bounds_ceil": ("chunk_bounds", _chunk_bounds_ceil),
    "shard_chunks_contiguous": ("shard_chunks", _shard_chunks_contiguous),
    "deal_wrong_local": ("interleave_deal", _deal_wrong_local),
    "deal_wrong_rank": ("interleave_deal", _deal_wrong_rank),
}


def _pins_fail():
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception:  # AssertionError, or a crash the mutation caused
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, fn)
    caught_by = _pins_fail()
    assert caught_by is not None, f"mutation {name} passed every pin"


def test_unmutated_oracle_passes_all_pins():
    assert _pins_fail() is None
