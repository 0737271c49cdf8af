"""Seeded random sweep of small shapes against the float64 oracle: varlen batches with ragged
lengths (including 1 and lengths below 2cp), cp in 1..8, query heads per kv head in 1..16,
head_dim 64 / 128, interleave sizes 1..16, for pass-KV (partials, merged and fused; plain and
over a contiguous cached context), pass-Q over paged round-robin caches, and decode (partials
and fused).  Each case is small enough for
the oracle; the sweep looks for edge cases the hand-picked cases miss."""
import math
import os
import random

import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_merged, check_partials

pytestmark = pytest.mark.gpu
DEV = "cuda"
# seeds per test; CPATTN_RANDOM_CASES widens the sweep (e.g. 80 for a long soak)
N_CASES = int(os.environ.get("CPATTN_RANDOM_CASES", "14"))


def _cu(lens):
    return torch.tensor([0] + torch.tensor(lens).cumsum(0).tolist(), dtype=torch.int32)


def _abs_v(t):
    """|V| (exact in bf16): the oracle's attention of it bounds the effect of P's bf16 rounding."""
    return t.abs()


def _rand_heads(r, max_g):
    Hkv = r.choice([1, 2, 4])
    G = r.randint(1, max_g)
    return G * Hkv, Hkv


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_pass_kv(lib, seed):
    r = random.Random(1000 + seed)
    B = r.randint(1, 3)
    cp = r.randint(1, 8)
    lens = [r.choice([1, r.randint(2, 2 * cp), r.randint(2, 700)]) for _ in range(B)]
    Hq, Hkv = _rand_heads(r, 8)
    d = r.choice([64, 128])
    x = wl.prefill_inputs(lens, Hq, Hkv, d, torch.bfloat16, seed=5000 + seed)
    q, k, v, cu = (x[n].to(DEV) for n in ("q", "k", "v", "cu_seqlens"))
    out, lse = lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=max(lens))
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Oa, _ = orc.pass_kv_partials(x["q"], x["k"], _abs_v(x["v"]), x["cu_seqlens"], cp, 1 / math.sqrt(d))
    what = f"pass-KV lens={lens} cp={cp} Hq/Hkv={Hq}/{Hkv} d={d}"
    check_partials(out, lse, O, L, what=what, o_abs=Oa)
    Om, Lm = orc.lse_merge(O, L)
    Oam, _ = orc.lse_merge(Oa, L)
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=torch.bfloat16)
    check_merged(mo, ml, Om, Lm, what=what + " merged", o_abs=Oam)
    fo, fl = lib.cp_attn_prefill_fused(q, cu, cp, k, v, max_seqlen_q=max(lens))
    check_merged(fo, fl, Om, Lm, what=what + " fused", o_abs=Oam)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_pass_kv_cached_context(lib, seed):
    r = random.Random(4000 + seed)
    B = r.randint(1, 3)
    cp = r.randint(1, 8)
    q_lens = [r.choice([0, 1, r.randint(2, 2 * cp), r.randint(2, 400)]) for _ in range(B)]
    kv_lens = [ql + r.choice([0, r.randint(1, 2 * cp), r.randint(1, 1200)]) for ql in q_lens]
    Hq, Hkv = _rand_heads(r, 8)
    d = r.choice([64, 128])
    g = torch.Generator().manual_seed(9000 + seed)
    qh = wl.normal((sum(q_lens), Hq, d), torch.bfloat16, g)
    kh = wl.normal((sum(kv_lens), Hkv, d), torch.bfloat16, g)
    vh = wl.normal((sum(kv_lens), Hkv, d), torch.bfloat16, g)
    cu, cu_kv = _cu(q_lens), _cu(kv_lens)
    what = f"pass-KV cached q={q_lens} kv={kv_lens} cp={cp} Hq/Hkv={Hq}/{Hkv} d={d}"
    if sum(q_lens) == 0:
        pytest.skip(what + ": no query rows")
    args = (qh.to(DEV), cu.to(DEV), cp)
    kw = dict(k=kh.to(DEV), v=vh.to(DEV), cu_seqlens_kv=cu_kv.to(DEV), max_seqlen_q=max(q_lens))
    out, lse = lib.cp_partial_attn_prefill(*args, **kw)
    O, L = orc.pass_kv_partials(qh, kh, vh, cu, cp, 1 / math.sqrt(d), cu_seqlens_kv=cu_kv)
    Oa, _ = orc.pass_kv_partials(qh, kh, _abs_v(vh), cu, cp, 1 / math.sqrt(d), cu_seqlens_kv=cu_kv)
    check_partials(out, lse, O, L, what=what, o_abs=Oa)
    Om, Lm = orc.lse_merge(O, L)
    Oam, _ = orc.lse_merge(Oa, L)
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=torch.bfloat16)
    check_merged(mo, ml, Om, Lm, what=what + " merged", o_abs=Oam)
    fo, fl = lib.cp_attn_prefill_fused(*args, **kw)
    check_merged(fo, fl, Om, Lm, what=what + " fused", o_abs=Oam)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_pass_q(lib, seed):
    r = random.Random(2000 + seed)
    B = r.randint(1, 3)
    cp = r.randint(1, 8)
    I = r.choice([1, 4, 8, 16])
    q_lens = [r.choice([1, r.randint(1, 300)]) for _ in range(B)]
    kv_lens = [ql + r.choice([0, r.randint(1, 1500)]) for ql in q_lens]
    Hq, Hkv = _rand_heads(r, 8)
    d = r.choice([64, 128])
    g = torch.Generator().manual_seed(6000 + seed)
    caps = [wl.block_capacity(L, cp, I, 16) for L in kv_lens]
    tables, pool = wl.shuffled_block_tables(caps, cp, g)
    kc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g)
    vc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g)
    qh = wl.normal((sum(q_lens), Hq, d), torch.bfloat16, g)
    cu = _cu(q_lens)
    sl = torch.tensor(kv_lens, dtype=torch.int32)
    out, lse = lib.cp_partial_attn_prefill(
        qh.to(DEV), cu.to(DEV), cp, mode=lib.CP_PASS_Q, k_cache=kc.to(DEV), v_cache=vc.to(DEV),
        block_tables=tables.to(DEV), seq_lens_kv=sl.to(DEV), interleave=I, max_seqlen_q=max(q_lens))
    O, L = orc.pass_q_partials(qh, kc, vc, tables, cu, sl, cp, I, 16, 1 / math.sqrt(d))
    Oa, _ = orc.pass_q_partials(qh, kc, _abs_v(vc), tables, cu, sl, cp, I, 16, 1 / math.sqrt(d))
    what = f"pass-Q q={q_lens} kv={kv_lens} cp={cp} I={I} Hq/Hkv={Hq}/{Hkv} d={d}"
    check_partials(out, lse, O, L, what=what, o_abs=Oa)
    Om, Lm = orc.lse_merge(O, L)
    Oam, _ = orc.lse_merge(Oa, L)
    fo, fl = lib.cp_attn_prefill_fused(
        qh.to(DEV), cu.to(DEV), cp, mode=lib.CP_PASS_Q, k_cache=kc.to(DEV), v_cache=vc.to(DEV),
        block_tables=tables.to(DEV), seq_lens_kv=sl.to(DEV), interleave=I, max_seqlen_q=max(q_lens))
    check_merged(fo, fl, Om, Lm, what=what + " fused", o_abs=Oam)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_decode(lib, seed):
    r = random.Random(3000 + seed)
    B = r.randint(1, 6)
    cp = r.randint(1, 8)
    I = r.choice([1, 2, 8, 16])
    lens = [r.choice([1, r.randint(1, 3 * cp * I), r.randint(1, 4000)]) for _ in range(B)]
    Hq, Hkv = _rand_heads(r, 16)
    d = r.choice([64, 128])
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, 7000 + seed,
                        8000 + seed, q_is_decode=True)
    dev = {n: x[n].to(DEV) for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    Oa, _ = orc.decode_partials(x["q"], x["k_cache"], _abs_v(x["v_cache"]), x["block_tables"],
                                x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Oam, _ = orc.lse_merge(Oa, L)
    what = f"decode lens={lens} cp={cp} I={I} Hq/Hkv={Hq}/{Hkv} d={d}"
    out, lse = lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"],
                                          dev["block_tables"], dev["seq_lens"], cp, I,
                                          max_seq_len=max(lens))
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=torch.bfloat16)
    check_merged(mo, ml, Om, Lm, what=what, o_abs=Oam)
    fo, fl = lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                     dev["block_tables"], dev["seq_lens"], cp, I,
                                     max_seq_len=max(lens))
    check_merged(fo, fl, Om, Lm, what=what + " fused", o_abs=Oam)
