"""Float64 reference definitions (test infrastructure; see the package docstring).

Notation: B sequences, Hq query heads, Hkv kv heads, G = Hq / Hkv query heads per
kv head (query head h reads kv head h // G), d head dim, cp logical ranks, I the
kv-cache interleave size, bs the page (block) size.  LSE is the natural log of
sum_j exp(scale * q . k_j) over the attended keys.

Inputs may be NumPy arrays or CPU torch tensors of any float dtype; every value is
upcast to float64 exactly as stored before any arithmetic.
"""
from __future__ import annotations

import numpy as np

_NEG_INF = -np.inf


def _f64(x):
    """Exact float64 copy of a NumPy array or CPU torch tensor (bf16 included)."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


# ----------------------------------------------------------------------------------------------
# Load-balanced prefill partition.
# "Add utility functions to enable pass-kv prefill and allgather decode", Purpose: during
# prefill both Q and KV are split over the CP ranks.  The split used here is the load-balanced
# one: 2*cp equal chunks (bounds floor(k*T/(2cp))), rank r holding chunk r and chunk 2cp-1-r.
# ----------------------------------------------------------------------------------------------

def chunk_bounds(T: int, cp: int) -> np.ndarray:
    """Chunk boundaries b_k = floor(k * T / (2 cp)), k = 0 .. 2cp (within one sequence)."""
    return np.array([(k * T) // (2 * cp) for k in range(2 * cp + 1)], dtype=np.int64)


def shard_chunks(r: int, cp: int):
    """The two chunks held by logical rank r, in storage order."""
    return (r, 2 * cp - 1 - r)


def partition(seq_lens, cp: int):
    """Token partition over cp logical ranks.

    Shard-major order: rank 0's rows first, then rank 1's, ...; inside a rank, sequence
    by sequence, and inside a sequence its chunk r before its chunk 2cp-1-r.

    Returns dict(perm, inv_perm, shard_offsets, chunk_bounds):
      perm[n]          global token index of shard-major row n   (int64 [N])
      inv_perm[t]      shard-major row of global token t          (int64 [N])
      shard_offsets[r] first shard-major row of rank r            (int64 [cp + 1])
      chunk_bounds     per-sequence chunk bounds (within-seq)     (int64 [B, 2cp + 1])
    """
    seq_lens = [int(x) for x in seq_lens]
    starts = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
    bounds = np.stack([chunk_bounds(T, cp) for T in seq_lens]) if seq_lens else \
        np.zeros((0, 2 * cp + 1), np.int64)
    perm = []
    shard_offsets = [0]
    for r in range(cp):
        for b, T in enumerate(seq_lens):
            for c in shard_chunks(r, cp):
                perm.extend(range(starts[b] + bounds[b, c], starts[b] + bounds[b, c + 1]))
        shard_offsets.append(len(perm))
    perm = np.array(perm, dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int64)
    return {"perm": perm, "inv_perm": inv, "shard_offsets": np.array(shard_offsets, np.int64),
            "chunk_bounds": bounds}


# ----------------------------------------------------------------------------------------------
# Round-robin kv placement.
# "Add utility functions ...", Purpose: for decode the KV tokens live on the CP ranks in a
# round-robin manner.  "[Feature] Prefill Context Parallel (PCP) basic support", code-review
# summary: the interleave size (how many consecutive tokens one rank takes before the turn
# passes on) is shared by prefill and decode CP; the GQA flashinfer page's Test Plan uses 8.
# Written as the deal itself: positions are dealt in groups of I, group g to rank g mod cp, and
# each rank stores what it receives in arrival order (local index = arrival count).
# ----------------------------------------------------------------------------------------------

def interleave_deal(L: int, cp: int, I: int):
    """Deal positions 0..L-1.  Returns (rank[L], local[L]) as int64 arrays."""
    p = np.arange(L, dtype=np.int64)
    rank = (p // I) % cp
    local = np.empty(L, dtype=np.int64)
    for r in range(cp):
        mine = rank == r
        local[mine] = np.arange(int(mine.sum()), dtype=np.int64)
    return rank, local


def rank_positions(L: int, r: int, cp: int, I: int) -> np.ndarray:
    """Global positions held by rank r, indexed by local index."""
    rank, _ = interleave_deal(L, cp, I)
    return np.nonzero(rank == r)[0].astype(np.int64)


def local_lengths(seq_lens, cp: int, I: int) -> np.ndarray:
    """Tokens each rank holds per sequence: int64 [cp, B]."""
    out = np.zeros((cp, len(seq_lens)), dtype=np.int64)
    for b, L in enumerate(seq_lens):
        rank, _ = interleave_deal(int(L), cp, I)
        for r in range(cp):
            out[r, b] = int((rank == r).sum())
    return out


def slot_mapping(seq_lens, cp: int, I: int, block_size: int, block_tables):
    """Where every token of every sequence lives (tokens concatenated sequence by sequence).

    Returns (rank[N], local[N], slot[N]) with slot = page * block_size + offset in the rank's
    own pool, page = block_tables[rank][b][local // block_size].
    """
    bt = _i64(block_tables)
    ranks, locs, slots = [], [], []
    for b, L in enumerate(seq_lens):
        rank, local = interleave_deal(int(L), cp, I)
        page = bt[rank, b, local // block_size]
        ranks.append(rank)
        locs.append(local)
        slots.append(page * block_size + local % block_size)
    cat = (lambda xs: np.concatenate(xs) if xs else np.zeros(0, np.int64))
    return cat(ranks), cat(locs), cat(slots)


def gather_rank_kv(cache_r, table_row, n_local: int, block_size: int):
    """Rank-local kv rows 0..n_local-1 of one sequence from a head-major page pool.

    cache_r: [pages, Hkv, block_size, d]; returns float64 [n_local, Hkv, d].
    """
    if n_local == 0:
        shape = cache_r.shape
        return np.zeros((0, shape[1], shape[3]), dtype=np.float64)
    loc = np.arange(n_local, dtype=np.int64)
    pages = _i64(table_row)[loc // block_size]
    offs = loc % block_size
    if hasattr(cache_r, "detach"):
        import torch
        rows = cache_r[torch.from_numpy(pages), :, torch.from_numpy(offs), :]
    else:
        rows = cache_r[pages, :, offs, :]
    return _f64(rows)


# ----------------------------------------------------------------------------------------------
# Attention and partial attention.
# "Add utility functions ...", Purpose: each token attends to every earlier token of its own
# sequence; with Q or KV sharded, each (Q shard, KV shard) pair yields a partial result that is
# merged later.  A partial is stored as (O_p, LSE_p): O_p normalised over its own key set and
# LSE_p = log sum exp of its scaled scores; an empty key set gives (0, -inf).
# ----------------------------------------------------------------------------------------------

def partial_attention(q, k, v, q_pos, k_pos, scale: float, row_block: int = 512):
    """Causal GQA attention of queries q over the key set (k, v).

    q: [Nq, Hq, d]; k, v: [Nk, Hkv, d]; q_pos [Nq], k_pos [Nk] absolute positions.
    Query i attends key j iff k_pos[j] <= q_pos[i].
    Returns O float64 [Nq, Hq, d] and LSE float64 [Nq, Hq].
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    q_pos = _i64(q_pos)
    k_pos = _i64(k_pos)
    Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[0], k.shape[1]
    G = Hq // Hkv
    O = np.zeros((Nq, Hq, d), dtype=np.float64)
    LSE = np.full((Nq, Hq), _NEG_INF, dtype=np.float64)
    if Nk == 0 or Nq == 0:
        return O, LSE
    for h in range(Hq):
        g = h // G
        kg = k[:, g, :]
        vg = v[:, g, :]
        for i0 in range(0, Nq, row_block):
            i1 = min(i0 + row_block, Nq)
            s = scale * (q[i0:i1, h, :] @ kg.T)                      # [n, Nk]
            visible = k_pos[None, :] <= q_pos[i0:i1, None]
            s = np.where(visible, s, _NEG_INF)
            m = s.max(axis=1)
            has = np.isfinite(m)
            e = np.zeros_like(s)
            e[has] = np.exp(s[has] - m[has, None])
            l = e.sum(axis=1)
            O[i0:i1, h, :][has] = (e[has] @ vg) / l[has, None]
            LSE[i0:i1, h][has] = m[has] + np.log(l[has])
    return O, LSE


def attention(q, k, v, scale: float, q_pos=None, k_pos=None):
    """Plain causal GQA attention of one sequence (default positions 0..N-1)."""
    Nq, Nk = q.shape[0], k.shape[0]
    if q_pos is None:
        q_pos = np.arange(Nk - Nq, Nk)
    if k_pos is None:
        k_pos = np.arange(Nk)
    return partial_attention(q, k, v, q_pos, k_pos, scale)


def lse_merge(O_parts, LSE_parts):
    """Merge P partials into exact attention.

    M = max_p LSE_p; w_p = exp(LSE_p - M) (0 for an empty partial); LSE = M + log sum_p w_p;
    O = sum_p w_p O_p / sum_p w_p, summed in order p = 0..P-1.  All partials empty gives
    (0, -inf).  Shapes: O_parts [P, ..., d], LSE_parts [P, ...].
    """
    O_parts = _f64(O_parts)
    LSE_parts = _f64(LSE_parts)
    M = LSE_parts.max(axis=0)
    fin = np.isfinite(M)
    w = np.zeros_like(LSE_parts)
    for p in range(LSE_parts.shape[0]):
        ok = np.isfinite(LSE_parts[p]) & fin
        w[p][ok] = np.exp(LSE_parts[p][ok] - M[ok])
    wsum = np.zeros_like(M)
    acc = np.zeros(O_parts.shape[1:], dtype=np.float64)
    for p in range(LSE_parts.shape[0]):
        wsum = wsum + w[p]
        # an empty partial has weight 0 and its stored O is never read
        contrib = np.where((w[p] > 0)[..., None], w[p][..., None] * np.nan_to_num(O_parts[p]), 0.0)
        acc = acc + contrib
    O = np.zeros_like(acc)
    O[fin] = acc[fin] / wsum[fin][..., None]
    LSE = np.full_like(M, _NEG_INF)
    LSE[fin] = M[fin] + np.log(wsum[fin])
    return O, LSE


# ----------------------------------------------------------------------------------------------
# The three CP flows, each a set of partials followed by lse_merge.
# ----------------------------------------------------------------------------------------------

def _rows_by_seq(cu, rows):
    """Split selected global rows (None = all) per sequence: list of within-seq index arrays."""
    cu = _i64(cu)
    B = cu.size - 1
    if rows is None:
        return [np.arange(cu[b + 1] - cu[b], dtype=np.int64) for b in range(B)]
    rows = np.asarray(rows, dtype=np.int64)
    out = []
    for b in range(B):
        sel = rows[(rows >= cu[b]) & (rows < cu[b + 1])]
        out.append(sel - cu[b])
    return out


def pass_kv_partials(q, k, v, cu_seqlens, cp: int, scale: float, rows=None, cu_seqlens_kv=None):
    """Pass-KV prefill: partial of every query row against every kv shard.

    "Add utility functions ...", Purpose: in full prefill the KV shards circulate so every Q
    shard meets every KV shard; the order of the rotation does not change any partial.
    Without cu_seqlens_kv, q, k and v hold the same tokens (self-attention, query i at
    position i).  With cu_seqlens_kv, sequence b has kv_len = cu_seqlens_kv[b+1] -
    cu_seqlens_kv[b] kv tokens (a cached context followed by the new tokens) and its q_len new
    queries are the last q_len positions: query i sits at position kv_len - q_len + i.  The kv
    tokens are cut into 2cp chunks exactly like the queries (chunk_bounds over kv_len) and kv
    shard s holds kv chunks s and 2cp-1-s.
    Returns O [cp, R, Hq, d], LSE [cp, R, Hq] where partial s is kv shard s and the R rows are
    the selected global query rows (all rows, in token order, when rows is None).
    """
    cu = _i64(cu_seqlens)
    cu_kv = cu if cu_seqlens_kv is None else _i64(cu_seqlens_kv)
    per_seq = _rows_by_seq(cu, rows)
    R = sum(x.size for x in per_seq)
    Hq, d = q.shape[1], q.shape[2]
    O = np.zeros((cp, R, Hq, d), dtype=np.float64)
    LSE = np.full((cp, R, Hq), _NEG_INF, dtype=np.float64)
    out_row = 0
    for b in range(cu.size - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        klo, khi = int(cu_kv[b]), int(cu_kv[b + 1])
        Tq, Tkv = hi - lo, khi - klo
        if Tkv < Tq:
            raise ValueError(f"sequence {b}: {Tkv} kv tokens for {Tq} new queries")
        ctx = Tkv - Tq
        sel = per_seq[b]
        if sel.size == 0:
            continue
        bnd = chunk_bounds(Tkv, cp)
        qb = q[lo:hi][sel]
        for s in range(cp):
            keys = np.concatenate([np.arange(bnd[c], bnd[c + 1]) for c in shard_chunks(s, cp)])
            kb = k[klo:khi][keys] if keys.size else k[klo:klo]
            vb = v[klo:khi][keys] if keys.size else v[klo:klo]
            o, l = partial_attention(qb, kb, vb, ctx + sel, keys, scale)
            O[s, out_row:out_row + sel.size] = o
            LSE[s, out_row:out_row + sel.size] = l
        out_row += sel.size
    return O, LSE


def pass_q_partials(q, k_cache, v_cache, block_tables, cu_seqlens_q, seq_lens_kv, cp: int,
                    I: int, block_size: int, scale: float, rows=None):
    """Pass-Q chunked prefill over a round-robin paged kv cache.

    "Add utility functions ...", Purpose: when the cached context is much longer than the new
    queries, the Q shards move and the KV stays where it is.  Sequence b has q_len new queries at
    positions kv_len - q_len .. kv_len - 1 and kv_len cached + new tokens dealt over the ranks
    (see interleave_deal).  Partial r = all selected query rows against rank r's resident keys.
    Returns O [cp, R, Hq, d], LSE [cp, R, Hq].
    """
    cu = _i64(cu_seqlens_q)
    kv_lens = _i64(seq_lens_kv)
    per_seq = _rows_by_seq(cu, rows)
    R = sum(x.size for x in per_seq)
    Hq, d = q.shape[1], q.shape[2]
    O = np.zeros((cp, R, Hq, d), dtype=np.float64)
    LSE = np.full((cp, R, Hq), _NEG_INF, dtype=np.float64)
    out_row = 0
    for b in range(cu.size - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        sel = per_seq[b]
        if sel.size == 0:
            continue
        L = int(kv_lens[b])
        ctx = L - (hi - lo)
        qb = q[lo:hi][sel]
        for r in range(cp):
            pos = rank_positions(L, r, cp, I)
            kr = gather_rank_kv(k_cache[r], block_tables[r][b], pos.size, block_size)
            vr = gather_rank_kv(v_cache[r], block_tables[r][b], pos.size, block_size)
            o, l = partial_attention(qb, kr, vr, ctx + sel, pos, scale)
            O[r, out_row:out_row + sel.size] = o
            LSE[r, out_row:out_row + sel.size] = l
        out_row += sel.size
    return O, LSE


def decode_partials(q, k_cache, v_cache, block_tables, seq_lens, cp: int, I: int,
                    block_size: int, scale: float, seqs=None):
    """Decode over a round-robin paged kv cache ("allgather decode").

    "Add utility functions ...", Purpose: decode KV stays round-robin on the CP ranks; the new
    query is made available to every rank, each rank attends over its own tokens and the
    partials are merged.  The query of sequence b sits at position L_b - 1 and its own kv entry
    is already in the cache.  Returns O [cp, B', Hq, d], LSE [cp, B', Hq] for the selected
    sequences (all when seqs is None).
    """
    lens = _i64(seq_lens)
    seqs = list(range(lens.size)) if seqs is None else list(seqs)
    Hq, d = q.shape[1], q.shape[2]
    O = np.zeros((cp, len(seqs), Hq, d), dtype=np.float64)
    LSE = np.full((cp, len(seqs), Hq), _NEG_INF, dtype=np.float64)
    for i, b in enumerate(seqs):
        L = int(lens[b])
        qb = q[b:b + 1]
        for r in range(cp):
            pos = rank_positions(L, r, cp, I)
            kr = gather_rank_kv(k_cache[r], block_tables[r][b], pos.size, block_size)
            vr = gather_rank_kv(v_cache[r], block_tables[r][b], pos.size, block_size)
            o, l = partial_attention(qb, kr, vr, np.array([L - 1]), pos, scale)
            O[r, i] = o[0]
            LSE[r, i] = l[0]
    return O, LSE


def kv_cache_write(k_new, v_new, cu_new, start_pos, cp: int, I: int, block_size: int,
                   block_tables, k_cache, v_cache):
    """Place new tokens' K/V rows into the per-rank head-major page pools (in place).

    "Add utility functions ...", Purpose (decode KV round-robin on the CP ranks) and "[Feature]
    Prefill Context Parallel (PCP) basic support", Purpose (per-rank block tables): sequence b's
    new rows cu_new[b]..cu_new[b+1]-1 sit at positions start_pos[b], start_pos[b]+1, ...; each
    goes to the rank and local index the round-robin deal gives its position, i.e. to page
    block_tables[rank][b][local // block_size], offset local % block_size.
    k_new, v_new: [N, Hkv, d]; k_cache, v_cache: [cp, pages, Hkv, block_size, d] (modified).
    """
    cu = _i64(cu_new)
    starts = _i64(start_pos)
    bt = _i64(block_tables)
    for b in range(cu.size - 1):
        n = int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        end = int(starts[b]) + n
        rank, local = interleave_deal(end, cp, I)
        for i in range(n):
            pos = int(starts[b]) + i
            r, l = int(rank[pos]), int(local[pos])
            page = int(bt[r, b, l // block_size])
            k_cache[r, page, :, l % block_size, :] = k_new[int(cu[b]) + i]
            v_cache[r, page, :, l % block_size, :] = v_new[int(cu[b]) + i]
