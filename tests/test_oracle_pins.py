"""Pins for the float64 oracle, independent of the oracle itself (CPU only).

Each check compares the oracle with something it does not share code with: a
pure-Python brute force on tiny inputs, torch's scaled_dot_product_attention (a
library routine) for plain causal attention, closed forms, invariants, and
hand-worked fixtures under tests/golden/.  ``test_oracle_mutations.py`` plants
mistakes in the oracle and checks that these pins catch them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import cp_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _read_kv_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [int(x) for x in v.split()]
    return out


# ---------------------------------------------------------------- brute force (pure Python)

def brute_attention(q, k, v, q_pos, k_pos, scale):
    """Scalar loops with math.exp / math.log; q [Nq][Hq][d], k/v [Nk][Hkv][d] as lists."""
    Nq, Hq, d = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k[0]) if k else 1
    G = Hq // Hkv
    O = [[[0.0] * d for _ in range(Hq)] for _ in range(Nq)]
    L = [[-math.inf] * Hq for _ in range(Nq)]
    for i in range(Nq):
        for h in range(Hq):
            g = h // G
            scores = []
            for j in range(len(k)):
                if k_pos[j] <= q_pos[i]:
                    dot = 0.0
                    for t in range(d):
                        dot += q[i][h][t] * k[j][g][t]
                    scores.append((j, scale * dot))
            if not scores:
                continue
            m = max(s for _, s in scores)
            z = sum(math.exp(s - m) for _, s in scores)
            L[i][h] = m + math.log(z)
            for j, s in scores:
                w = math.exp(s - m) / z
                for t in range(d):
                    O[i][h][t] += w * v[j][g][t]
    return np.array(O), np.array(L)


def pin_brute_force(seed=0):
    r = _rng(seed)
    for (Nq, Nk, Hq, Hkv, d, off) in [(7, 7, 4, 2, 5, 0), (5, 11, 4, 1, 3, 6), (1, 9, 2, 2, 4, 8),
                                     (6, 4, 6, 3, 2, -2)]:
        q = r.standard_normal((Nq, Hq, d))
        k = r.standard_normal((Nk, Hkv, d))
        v = r.standard_normal((Nk, Hkv, d))
        q_pos = np.arange(Nq) + off
        k_pos = np.arange(Nk)
        scale = 0.37
        O, L = orc.partial_attention(q, k, v, q_pos, k_pos, scale)
        Ob, Lb = brute_attention(q.tolist(), k.tolist(), v.tolist(), q_pos.tolist(),
                                 k_pos.tolist(), scale)
        assert np.array_equal(np.isinf(L), np.isinf(Lb))
        fin = np.isfinite(Lb)
        assert np.allclose(L[fin], Lb[fin], rtol=0, atol=1e-12)
        assert np.allclose(O, Ob, rtol=0, atol=1e-12)


def test_brute_force():
    pin_brute_force()


# ---------------------------------------------------------------- library routine (cp = 1)

def pin_sdpa(seed=1):
    r = _rng(seed)
    for (T, Hq, Hkv, d) in [(64, 8, 2, 16), (33, 4, 4, 8), (40, 6, 1, 12)]:
        q = r.standard_normal((T, Hq, d))
        k = r.standard_normal((T, Hkv, d))
        v = r.standard_normal((T, Hkv, d))
        scale = 1.0 / math.sqrt(d)
        O, L = orc.attention(q, k, v, scale)
        qt = torch.from_numpy(q).permute(1, 0, 2)[None]
        kt = torch.from_numpy(k).permute(1, 0, 2)[None]
        vt = torch.from_numpy(v).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, is_causal=True, scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
        assert np.allclose(O, ref.numpy(), rtol=0, atol=1e-12)
        # LSE from torch.logsumexp over the masked scores (heads expanded by repeat_interleave)
        ke = kt.repeat_interleave(Hq // Hkv, dim=1)
        s = torch.einsum("bhid,bhjd->bhij", qt, ke) * scale
        mask = torch.ones(T, T, dtype=torch.bool).tril()
        s = s.masked_fill(~mask, float("-inf"))
        lse = torch.logsumexp(s, dim=-1)[0].permute(1, 0)
        assert np.allclose(L, lse.numpy(), rtol=0, atol=1e-12)


def test_sdpa_cp1():
    pin_sdpa()


# ---------------------------------------------------------------- closed forms

def pin_closed_forms(seed=2):
    r = _rng(seed)
    T, Hq, Hkv, d = 24, 4, 2, 8
    scale = 0.5
    q = r.standard_normal((T, Hq, d))
    k = r.standard_normal((T, Hkv, d))
    # constant V -> O is that constant
    c = r.standard_normal(d)
    v = np.broadcast_to(c, (T, Hkv, d)).copy()
    O, L = orc.attention(q, k, v, scale)
    assert np.allclose(O, np.broadcast_to(c, O.shape), atol=1e-12)
    # all keys equal -> prefix mean of V, LSE = log(i+1) + scale q_i.k
    kk = np.broadcast_to(r.standard_normal((1, Hkv, d)), (T, Hkv, d)).copy()
    v = r.standard_normal((T, Hkv, d))
    O, L = orc.attention(q, kk, v, scale)
    G = Hq // Hkv
    for i in range(T):
        for h in range(Hq):
            g = h // G
            assert np.allclose(O[i, h], v[:i + 1, g].mean(axis=0), atol=1e-12)
            assert abs(L[i, h] - (math.log(i + 1) + scale * float(q[i, h] @ kk[0, g]))) < 1e-12
    # row 0 -> O = v_0, LSE = scale q_0.k_0
    O, L = orc.attention(q, k, v, scale)
    for h in range(Hq):
        g = h // G
        assert np.allclose(O[0, h], v[0, g], atol=1e-14)
        assert abs(L[0, h] - scale * float(q[0, h] @ k[0, g])) < 1e-12
    # GQA grouping: kv head g carries the constant value g -> q head h reads h // G
    vg = np.zeros((T, Hkv, d))
    for g in range(Hkv):
        vg[:, g, :] = g + 1.0
    Hq2, Hkv2 = 6, 3
    q2 = r.standard_normal((T, Hq2, d))
    k2 = r.standard_normal((T, Hkv2, d))
    v2 = np.zeros((T, Hkv2, d))
    for g in range(Hkv2):
        v2[:, g, :] = g + 1.0
    O, _ = orc.attention(q2, k2, v2, scale)
    for h in range(Hq2):
        assert np.allclose(O[:, h, :], h // (Hq2 // Hkv2) + 1.0, atol=1e-12)


def test_closed_forms():
    pin_closed_forms()


def pin_softmax_rows(seed=3):
    """V = identity makes O the attention weights: rows sum to 1, masked keys get exactly 0."""
    r = _rng(seed)
    T, Hq, Hkv = 20, 4, 2
    q = r.standard_normal((T, Hq, T))
    k = r.standard_normal((T, Hkv, T))
    v = np.broadcast_to(np.eye(T)[:, None, :], (T, Hkv, T)).copy()
    O, _ = orc.attention(q, k, v, 0.3)
    assert np.allclose(O.sum(axis=-1), 1.0, atol=1e-12)
    assert (O >= 0).all()
    for i in range(T):
        assert (O[i, :, i + 1:] == 0).all()
        assert (O[i, :, :i + 1] > 0).all()


def test_softmax_rows():
    pin_softmax_rows()


# ---------------------------------------------------------------- merge invariants

def pin_merge(seed=4):
    r = _rng(seed)
    P, R, H, d = 5, 7, 3, 4
    O = r.standard_normal((P, R, H, d))
    L = r.standard_normal((P, R, H)) * 3
    L[1, 2, 1] = -np.inf
    Om, Lm = orc.lse_merge(O, L)
    # permutation invariant
    perm = [3, 0, 4, 2, 1]
    Op, Lp = orc.lse_merge(O[perm], L[perm])
    assert np.allclose(Om, Op, atol=1e-12) and np.allclose(Lm, Lp, atol=1e-12)
    # empty partial is the identity
    Oe = np.concatenate([O, r.standard_normal((1, R, H, d))])
    Le = np.concatenate([L, np.full((1, R, H), -np.inf)])
    Ox, Lx = orc.lse_merge(Oe, Le)
    assert np.allclose(Om, Ox, atol=1e-12) and np.allclose(Lm, Lx, atol=1e-12)
    # two identical partials: O kept, LSE + ln 2
    O2, L2 = orc.lse_merge(np.stack([O[0], O[0]]), np.stack([L[0], L[0]]))
    fin = np.isfinite(L[0])
    assert np.allclose(O2[fin], O[0][fin], atol=1e-12)
    assert np.allclose(L2[fin], L[0][fin] + math.log(2), atol=1e-12)
    # associativity (also what makes split-kv decode exact)
    Oa, La = orc.lse_merge(O[:2], L[:2])
    Ob, Lb = orc.lse_merge(np.concatenate([Oa[None], O[2:]]), np.concatenate([La[None], L[2:]]))
    assert np.allclose(Om, Ob, atol=1e-12) and np.allclose(Lm, Lb, atol=1e-12)
    # all empty -> (0, -inf)
    Oz, Lz = orc.lse_merge(O[:2], np.full((2, R, H), -np.inf))
    assert (Oz == 0).all() and np.isneginf(Lz).all()
    # huge LSE values do not overflow
    Oh, Lh = orc.lse_merge(O[:2], np.stack([np.full((R, H), 800.0), np.full((R, H), 800.0)]))
    assert np.allclose(Lh, 800 + math.log(2)) and np.allclose(Oh, (O[0] + O[1]) / 2)
    # split of a key set: merging partials over a partition of the keys equals the whole
    T, Hq, Hkv, dd = 30, 4, 2, 6
    q = r.standard_normal((T, Hq, dd))
    k = r.standard_normal((T, Hkv, dd))
    v = r.standard_normal((T, Hkv, dd))
    Of, Lf = orc.attention(q, k, v, 0.4)
    sets = [np.array([0, 5, 9, 22]), np.array([1, 2, 3, 4, 6, 7, 8]),
            np.setdiff1d(np.arange(T), [0, 5, 9, 22, 1, 2, 3, 4, 6, 7, 8])]
    parts = [orc.partial_attention(q, k[s], v[s], np.arange(T), s, 0.4) for s in sets]
    Os, Ls = orc.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(Os, Of, atol=1e-12) and np.allclose(Ls, Lf, atol=1e-12)


def test_merge_invariants():
    pin_merge()


# ---------------------------------------------------------------- partition

def pin_partition_fixture():
    fx = _read_kv_fixture("partition_T10_cp2.txt")
    T, cp = fx["T"][0], fx["cp"][0]
    assert orc.chunk_bounds(T, cp).tolist() == fx["chunk_bounds"]
    part = orc.partition([T], cp)
    assert part["perm"].tolist() == fx["perm"]
    assert part["shard_offsets"].tolist() == fx["shard_offsets"]


def pin_partition_invariants():
    for lens, cp in [([256], 2), ([8192], 2), ([37, 5, 64, 1], 4), ([3], 4), ([100, 200], 8),
                     ([1, 2, 3, 17], 1), ([0, 9], 2)]:
        part = orc.partition(lens, cp)
        N = sum(lens)
        perm, inv = part["perm"], part["inv_perm"]
        assert sorted(perm.tolist()) == list(range(N))            # a permutation
        assert (inv[perm] == np.arange(N)).all()
        so = part["shard_offsets"]
        assert so[0] == 0 and so[-1] == N and (np.diff(so) >= 0).all()
        starts = np.concatenate([[0], np.cumsum(lens)])
        for b, T in enumerate(lens):
            bnd = part["chunk_bounds"][b]
            # 2cp chunks covering [0, T), sizes within one of each other
            assert bnd[0] == 0 and bnd[-1] == T
            sizes = np.diff(bnd)
            assert sizes.max() - sizes.min() <= 1
            for r in range(cp):
                rows = perm[so[r]:so[r + 1]]
                mine = rows[(rows >= starts[b]) & (rows < starts[b] + T)] - starts[b]
                want = list(range(bnd[r], bnd[r + 1])) + list(range(bnd[2 * cp - 1 - r],
                                                                     bnd[2 * cp - r]))
                assert mine.tolist() == want
        # every token is in exactly one shard
        owner = np.zeros(N, np.int64)
        for r in range(cp):
            owner[perm[so[r]:so[r + 1]]] += 1
        assert (owner == 1).all()


def pin_load_balance():
    """Per head, each shard's queries see 2cp c^2 + c visible (q, k) pairs (chunk size c).

    Counted through the oracle itself: with q = k = 0 every visible key has weight equal,
    so exp(LSE) is the number of visible keys of a row in that partial.
    """
    for cp in (1, 2, 4, 8):
        c = 3
        T = 2 * cp * c
        q = np.zeros((T, 1, 2))
        k = np.zeros((T, 1, 2))
        v = np.zeros((T, 1, 2))
        _, L = orc.pass_kv_partials(q, k, v, np.array([0, T]), cp, 1.0)
        counts = np.where(np.isfinite(L), np.exp(L), 0.0)          # [cp kv-shards, T, 1]
        part = orc.partition([T], cp)
        so = part["shard_offsets"]
        for r in range(cp):
            rows = part["perm"][so[r]:so[r + 1]]
            seen = counts[:, rows, 0].sum()
            assert abs(seen - (2 * cp * c * c + c)) < 1e-9, (cp, r, seen)


def test_partition():
    pin_partition_fixture()
    pin_partition_invariants()
    pin_load_balance()


# ---------------------------------------------------------------- interleave (round robin)

def brute_deal(L, cp, I):
    rank, local, count = [], [], [0] * cp
    owner, left = 0, I
    for _p in range(L):
        rank.append(owner)
        local.append(count[owner])
        count[owner] += 1
        left -= 1
        if left == 0:
            owner, left = (owner + 1) % cp, I
    return rank, local, count


def pin_interleave():
    fx = _read_kv_fixture("interleave_cp2_I8_L40.txt")
    rank, local = orc.interleave_deal(40, 2, 8)
    assert rank.tolist() == fx["rank"] and local.tolist() == fx["local"]
    assert orc.local_lengths([40], 2, 8)[:, 0].tolist() == fx["local_lengths"]
    for L in [0, 1, 7, 8, 9, 15, 16, 17, 100, 257, 1000]:
        for cp in (1, 2, 3, 4, 8):
            for I in (1, 2, 8, 16):
                rank, local = orc.interleave_deal(L, cp, I)
                br, bl, bc = brute_deal(L, cp, I)
                assert rank.tolist() == br and local.tolist() == bl
                lens = orc.local_lengths([L], cp, I)[:, 0]
                assert lens.tolist() == bc and lens.sum() == L
                # every position on exactly one rank, at a unique (rank, local)
                assert len(set(zip(rank.tolist(), local.tolist()))) == L
                for r in range(cp):
                    pos = orc.rank_positions(L, r, cp, I)
                    assert (np.diff(pos) > 0).all()
                    assert (rank[pos] == r).all() and (local[pos] == np.arange(pos.size)).all()
                if L % (I * cp) == 0:
                    assert (lens == L // cp).all()


def pin_computed_tokens_fixture():
    with open(os.path.join(GOLDEN, "computed_tokens_cp2.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    for cp, I, L, want in rows:
        assert orc.local_lengths([L], cp, I)[:, 0].tolist() == [want] * cp


def pin_slot_mapping(seed=5):
    g = torch.Generator().manual_seed(seed)
    lens, cp, I, bs = [37, 100, 1, 64], 2, 8, 16
    tables = torch.stack([torch.randperm(32, generator=g).to(torch.int32).view(4, 8)
                          for _ in range(cp)])
    rank, local, slot = orc.slot_mapping(lens, cp, I, bs, tables)
    assert len(set(zip(rank.tolist(), slot.tolist()))) == sum(lens)     # injective
    off = 0
    for b, L in enumerate(lens):
        br, bl, _ = brute_deal(L, cp, I)
        for p in range(L):
            n = off + p
            assert rank[n] == br[p] and local[n] == bl[p]
            assert slot[n] == int(tables[br[p], b, bl[p] // bs]) * bs + bl[p] % bs
        off += L


def test_interleave():
    pin_interleave()
    pin_computed_tokens_fixture()
    pin_slot_mapping()


# ---------------------------------------------------------------- sharded == unsharded

def _fill_pages(kc, vc, b, k_log, v_log, cp, I, bs, tables):
    br, bl, _ = brute_deal(k_log.shape[0], cp, I)
    for p in range(k_log.shape[0]):
        page = int(tables[br[p], b, bl[p] // bs])
        kc[br[p], page, :, bl[p] % bs, :] = k_log[p]
        vc[br[p], page, :, bl[p] % bs, :] = v_log[p]


def pin_pass_kv_equals_attention(seed=6):
    r = _rng(seed)
    lens = [13, 40, 5, 1]
    Hq, Hkv, d = 4, 2, 8
    N = sum(lens)
    q = r.standard_normal((N, Hq, d))
    k = r.standard_normal((N, Hkv, d))
    v = r.standard_normal((N, Hkv, d))
    cu = np.concatenate([[0], np.cumsum(lens)])
    for cp in (1, 2, 4, 8):
        O, L = orc.pass_kv_partials(q, k, v, cu, cp, 0.3)
        Om, Lm = orc.lse_merge(O, L)
        for b in range(len(lens)):
            sl = slice(cu[b], cu[b + 1])
            Of, Lf = orc.attention(q[sl], k[sl], v[sl], 0.3)
            assert np.allclose(Om[sl], Of, atol=1e-12), cp
            assert np.allclose(Lm[sl], Lf, atol=1e-12), cp
        if cp == 1:
            assert np.allclose(O[0], Om, atol=1e-14)
    # sampled rows give the same values as the full computation
    rows = [0, 3, 12, 13, 30, 52, 57]
    O, L = orc.pass_kv_partials(q, k, v, cu, 4, 0.3)
    Os, Ls = orc.pass_kv_partials(q, k, v, cu, 4, 0.3, rows=rows)
    assert np.allclose(Os, O[:, rows], atol=1e-12) and np.allclose(Ls, L[:, rows], atol=1e-12)


def pin_pass_kv_cached_context(seed=16):
    """Pass-KV over a cached context (queries = the last q_len of kv_len positions): merged
    partials equal torch's scaled_dot_product_attention with an explicit bottom-right causal
    mask (key j visible to new query i iff j <= kv_len - q_len + i) for cp in {1, 2, 4, 8};
    with kv_len = q_len the partials equal those of plain self-attention; a brute-force loop
    checks one tiny case end to end."""
    r = _rng(seed)
    q_lens, kv_lens = [5, 17, 1, 9], [37, 17, 30, 9]
    Hq, Hkv, d = 4, 2, 8
    q = r.standard_normal((sum(q_lens), Hq, d))
    k = r.standard_normal((sum(kv_lens), Hkv, d))
    v = r.standard_normal((sum(kv_lens), Hkv, d))
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    cu_kv = np.concatenate([[0], np.cumsum(kv_lens)])
    for cp in (1, 2, 4, 8):
        O, L = orc.pass_kv_partials(q, k, v, cu, cp, 0.3, cu_seqlens_kv=cu_kv)
        Om, Lm = orc.lse_merge(O, L)
        for b in range(len(q_lens)):
            sq, sk = slice(cu[b], cu[b + 1]), slice(cu_kv[b], cu_kv[b + 1])
            nq, nk = q_lens[b], kv_lens[b]
            mask = torch.from_numpy(np.arange(nk)[None, :] <= (nk - nq + np.arange(nq))[:, None])
            qt = torch.from_numpy(q[sq]).permute(1, 0, 2)[None]
            kt = torch.from_numpy(k[sk]).permute(1, 0, 2)[None].repeat_interleave(Hq // Hkv, 1)
            vt = torch.from_numpy(v[sk]).permute(1, 0, 2)[None].repeat_interleave(Hq // Hkv, 1)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, attn_mask=mask, scale=0.3)[0].permute(1, 0, 2).numpy()
            s_ = (torch.einsum("bhid,bhjd->bhij", qt, kt) * 0.3).masked_fill(~mask, float("-inf"))
            lse = torch.logsumexp(s_, dim=-1)[0].permute(1, 0).numpy()
            assert np.allclose(Om[sq], ref, atol=1e-12), (cp, b)
            assert np.allclose(Lm[sq], lse, atol=1e-12), (cp, b)
    # kv_len = q_len: the same partials as the self-attention form
    lens = [11, 6]
    qs = r.standard_normal((17, Hq, d))
    ks = r.standard_normal((17, Hkv, d))
    vs = r.standard_normal((17, Hkv, d))
    cs = np.array([0, 11, 17])
    O1, L1 = orc.pass_kv_partials(qs, ks, vs, cs, 2, 0.3)
    O2, L2 = orc.pass_kv_partials(qs, ks, vs, cs, 2, 0.3, cu_seqlens_kv=cs)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # brute force: one sequence, 3 new queries after 6 cached tokens, cp = 2 (chunks of 2 and
    # 3 kv tokens: bounds 0, 2, 4, 6, 9 over kv_len = 9 -> shard 0 = {0, 1, 6, 7, 8})
    qb = r.standard_normal((3, 2, 3))
    kb = r.standard_normal((9, 1, 3))
    vb = r.standard_normal((9, 1, 3))
    O, L = orc.pass_kv_partials(qb, kb, vb, np.array([0, 3]), 2, 0.7,
                                cu_seqlens_kv=np.array([0, 9]))
    for s_, keys in ((0, [0, 1, 6, 7, 8]), (1, [2, 3, 4, 5])):
        Ob, Lb = brute_attention(qb.tolist(), kb[keys].tolist(), vb[keys].tolist(),
                                 [6, 7, 8], keys, 0.7)
        assert np.array_equal(np.isinf(L[s_]), np.isinf(Lb))
        fin = np.isfinite(Lb)
        assert np.allclose(L[s_][fin], Lb[fin], atol=1e-12) and np.allclose(O[s_], Ob, atol=1e-12)
    # sampled rows give the same values as the full computation
    rows = [0, 4, 5, 21, 22, 31]
    O, L = orc.pass_kv_partials(q, k, v, cu, 4, 0.3, cu_seqlens_kv=cu_kv)
    Os, Ls = orc.pass_kv_partials(q, k, v, cu, 4, 0.3, rows=rows, cu_seqlens_kv=cu_kv)
    assert np.allclose(Os, O[:, rows], atol=1e-12) and np.allclose(Ls, L[:, rows], atol=1e-12)


def test_pass_kv_cached_context():
    pin_pass_kv_cached_context()


def pin_pass_q_equals_attention(seed=7):
    r = _rng(seed)
    Hq, Hkv, d, bs = 4, 2, 8, 4
    kv_lens = [45, 19, 64]
    q_lens = [7, 19, 3]
    for cp, I in [(1, 8), (2, 8), (4, 2), (8, 1), (3, 4)]:
        caps = [-(-L // bs) for L in kv_lens]
        pool = sum(caps)
        g = torch.Generator().manual_seed(seed + cp)
        tables = np.full((cp, len(kv_lens), max(caps)), -1, np.int64)
        for rr in range(cp):
            perm = torch.randperm(pool, generator=g).numpy()
            off = 0
            for b, c in enumerate(caps):
                tables[rr, b, :c] = perm[off:off + c]
                off += c
        kc = np.full((cp, pool, Hkv, bs, d), np.nan)
        vc = np.full((cp, pool, Hkv, bs, d), np.nan)
        logical = []
        for b, L in enumerate(kv_lens):
            kl = r.standard_normal((L, Hkv, d))
            vl = r.standard_normal((L, Hkv, d))
            _fill_pages(kc, vc, b, kl, vl, cp, I, bs, tables)
            logical.append((kl, vl))
        cu_q = np.concatenate([[0], np.cumsum(q_lens)])
        q = r.standard_normal((cu_q[-1], Hq, d))
        O, L = orc.pass_q_partials(q, kc, vc, tables, cu_q, kv_lens, cp, I, bs, 0.25)
        Om, Lm = orc.lse_merge(O, L)
        for b, Lkv in enumerate(kv_lens):
            sl = slice(cu_q[b], cu_q[b + 1])
            kl, vl = logical[b]
            Of, Lf = orc.attention(q[sl], kl, vl, 0.25)
            assert np.allclose(Om[sl], Of, atol=1e-12), (cp, I, b)
            assert np.allclose(Lm[sl], Lf, atol=1e-12), (cp, I, b)
        # decode: one query per sequence at position L - 1
        qd = r.standard_normal((len(kv_lens), Hq, d))
        Od, Ld = orc.decode_partials(qd, kc, vc, tables, kv_lens, cp, I, bs, 0.25)
        Odm, Ldm = orc.lse_merge(Od, Ld)
        for b, Lkv in enumerate(kv_lens):
            kl, vl = logical[b]
            Of, Lf = orc.attention(qd[b:b + 1], kl, vl, 0.25)
            assert np.allclose(Odm[b], Of[0], atol=1e-12), (cp, I, b)
            assert np.allclose(Ldm[b], Lf[0], atol=1e-12), (cp, I, b)


def test_sharded_equals_unsharded():
    pin_pass_kv_equals_attention()
    pin_pass_q_equals_attention()


def pin_kv_cache_write(seed=8):
    """Tokens written in several pieces land where a pure-Python deal says (round trip through
    the gather that the pass-Q and decode flows use gives back the logical rows)."""
    r = _rng(seed)
    Hkv, d, bs, cp, I = 2, 4, 4, 3, 2
    L = [23, 9]
    caps = [-(-x // bs) + 2 for x in L]
    pool = sum(caps)
    tables = np.full((cp, 2, max(caps)), -1, np.int64)
    for rr in range(cp):
        perm = r.permutation(pool)
        off = 0
        for b, c in enumerate(caps):
            tables[rr, b, :c] = perm[off:off + c]
            off += c
    kc = np.full((cp, pool, Hkv, bs, d), np.nan)
    vc = np.full((cp, pool, Hkv, bs, d), np.nan)
    logical = [(r.standard_normal((x, Hkv, d)), r.standard_normal((x, Hkv, d))) for x in L]
    pieces = [(0, 10, 0, 4), (10, 23, 4, 9)]   # (start, end) per sequence in two writes
    for (s0, e0, s1, e1) in pieces:
        kn = np.concatenate([logical[0][0][s0:e0], logical[1][0][s1:e1]])
        vn = np.concatenate([logical[0][1][s0:e0], logical[1][1][s1:e1]])
        cu = np.array([0, e0 - s0, e0 - s0 + e1 - s1])
        orc.kv_cache_write(kn, vn, cu, np.array([s0, s1]), cp, I, bs, tables, kc, vc)
    for b, x in enumerate(L):
        br, bl, _ = brute_deal(x, cp, I)
        for p in range(x):
            page = tables[br[p], b, bl[p] // bs]
            assert np.array_equal(kc[br[p], page, :, bl[p] % bs], logical[b][0][p])
            assert np.array_equal(vc[br[p], page, :, bl[p] % bs], logical[b][1][p])
        for rr in range(cp):
            pos = orc.rank_positions(x, rr, cp, I)
            kg = orc.gather_rank_kv(kc[rr], tables[rr, b], pos.size, bs)
            assert np.array_equal(kg, logical[b][0][pos])


def test_kv_cache_write():
    pin_kv_cache_write()


ALL_PINS = [pin_brute_force, pin_kv_cache_write, pin_sdpa, pin_closed_forms, pin_softmax_rows, pin_merge,
            pin_partition_fixture, pin_partition_invariants, pin_load_balance, pin_interleave,
            pin_computed_tokens_fixture, pin_slot_mapping, pin_pass_kv_equals_attention,
            pin_pass_kv_cached_context, pin_pass_q_equals_attention]


@pytest.mark.parametrize("T,cp", [(4, 2), (2, 4), (1, 8)])
def test_tiny_edge_cases(T, cp):
    """Sequences shorter than 2cp: some chunks are empty; results still exact."""
    r = _rng(T * 10 + cp)
    q = r.standard_normal((T, 2, 4))
    k = r.standard_normal((T, 1, 4))
    v = r.standard_normal((T, 1, 4))
    O, L = orc.pass_kv_partials(q, k, v, np.array([0, T]), cp, 0.5)
    Om, Lm = orc.lse_merge(O, L)
    Of, Lf = orc.attention(q, k, v, 0.5)
    assert np.allclose(Om, Of, atol=1e-12) and np.allclose(Lm, Lf, atol=1e-12)
