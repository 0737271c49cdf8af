"""GPU parity: every C-ABI entry point against the float64 oracle on the same seeded inputs.

Small cases span several tiles and ragged tails; index maps are compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_merged, check_partials, check_same_rounded, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _cu(lens):
    cu = [0]
    for x in lens:
        cu.append(cu[-1] + x)
    return torch.tensor(cu, dtype=torch.int32)


# ------------------------------------------------------------------------------------ maps

@pytest.mark.parametrize("lens,cp", [([256], 2), ([8192], 2), ([32768, 32768], 4), ([37, 5, 64, 1], 4),
                                     ([3], 4), ([100, 200, 0, 7], 8), ([1, 2, 3, 17], 1),
                                     ([2048] * 4, 4), ([1000] * 37, 3)])
def test_partition_bitexact(lib, lens, cp):
    cu = _cu(lens)
    perm, inv, so, cb = lib.cp_partition(cu.to(DEV), cp, sum(lens))
    ref = orc.partition(lens, cp)
    assert perm.cpu().numpy().tolist() == ref["perm"].tolist()
    assert inv.cpu().numpy().tolist() == ref["inv_perm"].tolist()
    assert so.cpu().numpy().tolist() == ref["shard_offsets"].tolist()
    assert cb.cpu().numpy().tolist() == ref["chunk_bounds"].tolist()


@pytest.mark.parametrize("lens,cp,I", [([40], 2, 8), ([37, 100, 1, 64], 2, 8), ([32768] * 4, 4, 8),
                                       ([1023, 5000, 16], 3, 4), ([77], 8, 1), ([9, 130], 1, 16)])
def test_interleave_bitexact(lib, lens, cp, I):
    bs = 16
    caps = [wl.block_capacity(L, cp, I, bs) for L in lens]
    tables, pool = wl.shuffled_block_tables(caps, cp, torch.Generator().manual_seed(7))
    cu = _cu(lens)
    ll, rk, lc, sl = lib.cp_kv_interleave_layout(cu.to(DEV), cp, I, sum(lens), bs,
                                                 block_tables=tables.to(DEV))
    rank, local, slot = orc.slot_mapping(lens, cp, I, bs, tables)
    assert ll.cpu().numpy().tolist() == orc.local_lengths(lens, cp, I).tolist()
    assert rk.cpu().numpy().tolist() == rank.tolist()
    assert lc.cpu().numpy().tolist() == local.tolist()
    assert sl.cpu().numpy().tolist() == slot.tolist()


def test_interleave_reports_bad_table(lib):
    lens, cp, I = [64], 2, 8
    tables = torch.full((cp, 1, 1), 3, dtype=torch.int32)   # one column: too short for 32 tokens
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, _, sl = lib.cp_kv_interleave_layout(_cu(lens).to(DEV), cp, I, 64, 16,
                                              block_tables=tables.to(DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    assert (sl.cpu() == -1).sum().item() == 32


# ------------------------------------------------------------------------------------ merge

@pytest.mark.parametrize("P,rows,H,d,dt", [(2, 1000, 16, 128, torch.bfloat16), (5, 77, 3, 64, torch.float32),
                                           (64, 33, 32, 128, torch.bfloat16), (1, 9, 2, 128, torch.float32)])
def test_merge_parity(lib, P, rows, H, d, dt):
    g = torch.Generator().manual_seed(P * 1000 + rows)
    O = torch.randn(P, rows, H, d, generator=g)
    L = torch.randn(P, rows, H, generator=g) * 4
    L[torch.rand(P, rows, H, generator=g) < 0.3] = -math.inf   # empty partials
    L[:, 0, 0] = -math.inf                                      # a fully empty unit
    O[torch.isinf(L)] = float("nan")                            # never read when empty
    out, lse = lib.cp_lse_merge(O.to(DEV), L.to(DEV), out_dtype=dt)
    Or, Lr = orc.lse_merge(O.numpy(), L.numpy())
    # the merge alone is exact up to f32 rounding; a bf16 output adds at most half an ulp
    # (2^-9 |O|).  Random partials here reach |O| ~ 4, so the bound is relative.
    ref = torch.from_numpy(Or)
    tol = (2.0 ** -8 if dt == torch.bfloat16 else 1e-5) * ref.abs() + 1e-5
    assert ((out.double().cpu() - ref).abs() <= tol).all(), "merge output"
    fin = torch.isfinite(torch.from_numpy(Lr))
    assert torch.equal(torch.isfinite(lse.cpu()), fin)
    assert ((lse.double().cpu()[fin] - torch.from_numpy(Lr)[fin]).abs()
            <= 1e-5 * torch.from_numpy(Lr)[fin].abs() + 1e-5).all(), "merge lse"


# ------------------------------------------------------------------------------------ prefill

def _impl_code(lib, name):
    return {"simt": lib.CP_IMPL_SIMT, "tc": lib.CP_IMPL_TCGEN05,
            "tc1": lib.CP_IMPL_TCGEN05_SINGLE}[name]


PASS_KV_CASES = [
    # lens, Hq, Hkv, d, dtype, cp
    ([256], 4, 1, 64, torch.float32, 2),          # the tiny workload
    ([1000, 333, 1], 8, 2, 128, torch.bfloat16, 2),
    ([700, 129], 16, 2, 128, torch.bfloat16, 4),
    ([515], 4, 4, 64, torch.bfloat16, 3),
    ([300, 5], 8, 1, 128, torch.bfloat16, 8),
    ([640], 8, 2, 128, torch.float32, 1),
    ([4096], 16, 2, 128, torch.bfloat16, 2),      # ~512 work items: several waves of CTAs
    ([777, 64], 8, 2, 64, torch.bfloat16, 2),     # two-head kernel at d = 64, ragged tiles
]


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
@pytest.mark.parametrize("case", range(len(PASS_KV_CASES)))
def test_pass_kv_parity(lib, case, impl):
    lens, Hq, Hkv, d, dt, cp = PASS_KV_CASES[case]
    if impl.startswith("tc") and dt != torch.bfloat16:
        pytest.skip("the tensor-core kernel takes bf16")
    x = wl.prefill_inputs(lens, Hq, Hkv, d, dt, seed=100 + case)
    scale = 1.0 / math.sqrt(d)
    out, lse = lib.cp_partial_attn_prefill(
        x["q"].to(DEV), x["cu_seqlens"].to(DEV), cp, k=x["k"].to(DEV), v=x["v"].to(DEV),
        max_seqlen_q=max(lens), impl=_impl_code(lib, impl))
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, scale)
    check_partials(out, lse, O, L, what=f"pass-KV {impl} partials")
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=dt)
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what=f"pass-KV {impl} merged")


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
def test_pass_kv_single_pair(lib, impl):
    """q_shard / kv_shard restrict the launch to one rotation step; other pairs untouched."""
    lens, Hq, Hkv, d, cp = [900], 8, 2, 128, 4
    x = wl.prefill_inputs(lens, Hq, Hkv, d, torch.bfloat16, seed=55)
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    part = orc.partition(lens, cp)
    out = torch.full((cp, 900, Hq, d), 7.0, device=DEV)
    lse = torch.full((cp, 900, Hq), 7.0, device=DEV)
    qs, ks = 1, 2
    lib.cp_partial_attn_prefill(x["q"].to(DEV), x["cu_seqlens"].to(DEV), cp, k=x["k"].to(DEV),
                                v=x["v"].to(DEV), q_shard=qs, kv_shard=ks, out=out, lse=lse,
                                impl=_impl_code(lib, impl), max_seqlen_q=900)
    rows = part["perm"][part["shard_offsets"][qs]:part["shard_offsets"][qs + 1]]
    check_partials(out[ks:ks + 1], lse[ks:ks + 1], O[ks:ks + 1][:, rows], L[ks:ks + 1][:, rows],
                   rows=rows.tolist(), what="single pair")
    mask = torch.ones(cp, 900, dtype=torch.bool)
    mask[ks, torch.as_tensor(rows)] = False
    assert (lse.cpu()[mask] == 7.0).all()


PASS_KV_CTX_CASES = [
    # q_lens, kv_lens (cached + new), Hq, Hkv, d, dtype, cp
    ([300, 77], [1500, 77], 8, 2, 128, torch.bfloat16, 2),    # one cached, one plain sequence
    ([512, 1, 130], [4096, 900, 131], 16, 2, 128, torch.bfloat16, 4),
    ([200], [2000], 6, 2, 64, torch.bfloat16, 3),             # odd G: two row tiles per CTA
    ([129, 0, 64], [700, 50, 64], 4, 1, 128, torch.bfloat16, 1),   # a sequence with no query
    ([96], [1000], 8, 2, 128, torch.float32, 2),
]


def _ctx_case(q_lens, kv_lens, Hq, Hkv, d, dt, seed):
    g = torch.Generator().manual_seed(seed)
    return dict(q=wl.normal((sum(q_lens), Hq, d), dt, g), k=wl.normal((sum(kv_lens), Hkv, d), dt, g),
                v=wl.normal((sum(kv_lens), Hkv, d), dt, g), cu_q=_cu(q_lens), cu_kv=_cu(kv_lens))


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
@pytest.mark.parametrize("case", range(len(PASS_KV_CTX_CASES)))
def test_pass_kv_cached_context_parity(lib, case, impl):
    """Pass-KV with a contiguous cached context (cu_seqlens_kv): the new queries are the last
    positions of their sequence's kv tokens, kv shards cut over the kv length."""
    q_lens, kv_lens, Hq, Hkv, d, dt, cp = PASS_KV_CTX_CASES[case]
    if impl.startswith("tc") and dt != torch.bfloat16:
        pytest.skip("the tensor-core kernel takes bf16")
    x = _ctx_case(q_lens, kv_lens, Hq, Hkv, d, dt, 500 + case)
    out, lse = lib.cp_partial_attn_prefill(
        x["q"].to(DEV), x["cu_q"].to(DEV), cp, k=x["k"].to(DEV), v=x["v"].to(DEV),
        cu_seqlens_kv=x["cu_kv"].to(DEV), max_seqlen_q=max(q_lens), impl=_impl_code(lib, impl))
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_q"], cp, 1 / math.sqrt(d),
                                cu_seqlens_kv=x["cu_kv"])
    check_partials(out, lse, O, L, what=f"pass-KV cached context {impl} partials")
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=dt)
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what=f"pass-KV cached context {impl} merged")
    if dt == torch.bfloat16 and impl != "simt":
        fo, fl = lib.cp_attn_prefill_fused(x["q"].to(DEV), x["cu_q"].to(DEV), cp, x["k"].to(DEV),
                                           x["v"].to(DEV), cu_seqlens_kv=x["cu_kv"].to(DEV),
                                           max_seqlen_q=max(q_lens), impl=_impl_code(lib, impl))
        check_merged(fo, fl, Om, Lm, what=f"pass-KV cached context {impl} fused")


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
def test_pass_kv_cached_context_single_pair(lib, impl):
    """One rotation step over a cached context: q_shard / kv_shard select one (Q shard, KV shard)
    pair, the KV shard cut over the kv length; the other pairs' outputs stay untouched."""
    q_lens, kv_lens, Hq, Hkv, d, cp = [300], [1700], 8, 2, 128, 3
    x = _ctx_case(q_lens, kv_lens, Hq, Hkv, d, torch.bfloat16, 91)
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_q"], cp, 1 / math.sqrt(d),
                                cu_seqlens_kv=x["cu_kv"])
    part = orc.partition(q_lens, cp)
    out = torch.full((cp, 300, Hq, d), 7.0, device=DEV)
    lse = torch.full((cp, 300, Hq), 7.0, device=DEV)
    qs, ks = 2, 1
    lib.cp_partial_attn_prefill(x["q"].to(DEV), x["cu_q"].to(DEV), cp, k=x["k"].to(DEV),
                                v=x["v"].to(DEV), cu_seqlens_kv=x["cu_kv"].to(DEV), q_shard=qs,
                                kv_shard=ks, out=out, lse=lse, impl=_impl_code(lib, impl),
                                max_seqlen_q=300)
    rows = part["perm"][part["shard_offsets"][qs]:part["shard_offsets"][qs + 1]]
    check_partials(out[ks:ks + 1], lse[ks:ks + 1], O[ks:ks + 1][:, rows], L[ks:ks + 1][:, rows],
                   rows=rows.tolist(), what=f"cached-context single pair {impl}")
    mask = torch.ones(cp, 300, dtype=torch.bool)
    mask[ks, torch.as_tensor(rows)] = False
    assert (lse.cpu()[mask] == 7.0).all()


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
def test_pass_kv_reports_short_kv(lib, impl):
    """A sequence with fewer kv tokens than new queries is flagged (CP_ERR_DEVICE_BOUNDS) and its
    rows skipped; the other sequences' partials still match the oracle."""
    q_lens, kv_lens = [40, 30], [100, 20]      # sequence 1: 20 kv tokens for 30 queries
    x = _ctx_case(q_lens, kv_lens, 8, 2, 128, torch.bfloat16, 77)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.cp_partial_attn_prefill(
        x["q"].to(DEV), x["cu_q"].to(DEV), 2, k=x["k"].to(DEV), v=x["v"].to(DEV),
        cu_seqlens_kv=x["cu_kv"].to(DEV), max_seqlen_q=40, impl=_impl_code(lib, impl), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    O, L = orc.pass_kv_partials(x["q"][:40], x["k"][:100], x["v"][:100], _cu([40]), 2, 1 / math.sqrt(128),
                                cu_seqlens_kv=_cu([100]))
    check_partials(out[:, :40], lse[:, :40], O, L, what=f"pass-KV {impl} beside a flagged sequence")


def _paged_case(B, q_lens, kv_lens, Hq, Hkv, d, dt, cp, I, seed):
    g = torch.Generator().manual_seed(seed)
    caps = [wl.block_capacity(L, cp, I, 16) for L in kv_lens]
    tables, pool = wl.shuffled_block_tables(caps, cp, torch.Generator().manual_seed(seed + 1))
    q = wl.normal((sum(q_lens), Hq, d), dt, g)
    kc = wl.normal((cp, pool, Hkv, 16, d), dt, g)
    vc = wl.normal((cp, pool, Hkv, 16, d), dt, g)
    return dict(q=q, k_cache=kc, v_cache=vc, block_tables=tables, cu_seqlens_q=_cu(q_lens),
                seq_lens=torch.tensor(kv_lens, dtype=torch.int32))


PASS_Q_CASES = [
    # q_lens, kv_lens, Hq, Hkv, d, dtype, cp, I
    ([100, 37], [700, 300], 8, 2, 128, torch.bfloat16, 4, 8),
    ([256], [256], 16, 2, 128, torch.bfloat16, 2, 8),          # no cached context
    ([130, 1, 64], [1000, 1, 64], 4, 1, 64, torch.bfloat16, 3, 4),
    ([50], [2000], 8, 8, 128, torch.float32, 2, 16),
    ([200], [1500], 8, 2, 128, torch.bfloat16, 1, 8),
    ([512, 512], [4096, 3000], 16, 2, 128, torch.bfloat16, 4, 8),   # ~512 work items
    # fused: 192 items, so more than one wave on 152 SMs with a split tail
    ([1024, 1024, 1024], [4096, 3500, 1100], 16, 2, 128, torch.bfloat16, 4, 8),
]


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
@pytest.mark.parametrize("case", range(len(PASS_Q_CASES)))
def test_pass_q_parity(lib, case, impl):
    q_lens, kv_lens, Hq, Hkv, d, dt, cp, I = PASS_Q_CASES[case]
    if impl.startswith("tc") and dt != torch.bfloat16:
        pytest.skip("the tensor-core kernel takes bf16")
    x = _paged_case(len(q_lens), q_lens, kv_lens, Hq, Hkv, d, dt, cp, I, 300 + case)
    out, lse = lib.cp_partial_attn_prefill(
        x["q"].to(DEV), x["cu_seqlens_q"].to(DEV), cp, mode=lib.CP_PASS_Q,
        k_cache=x["k_cache"].to(DEV), v_cache=x["v_cache"].to(DEV),
        block_tables=x["block_tables"].to(DEV), seq_lens_kv=x["seq_lens"].to(DEV), interleave=I,
        max_seqlen_q=max(q_lens), impl=_impl_code(lib, impl))
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    check_partials(out, lse, O, L, what=f"pass-Q {impl} partials")
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=dt)
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what=f"pass-Q {impl} merged")


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
def test_pass_q_reports_bad_page(lib, impl):
    """Block-table entries outside the pool (too large, negative) are checked before any read:
    the kernel flags CP_ERR_DEVICE_BOUNDS and the next valid call still matches the oracle."""
    x = _paged_case(1, [20], [300], 4, 1, 64, torch.bfloat16, 2, 8, 9)
    dev = {n: x[n].to(DEV) for n in ("q", "cu_seqlens_q", "k_cache", "v_cache", "seq_lens")}
    tables = x["block_tables"].clone()
    tables[1, 0, 1] = 10 ** 6          # outside the pool
    tables[0, 0, 3] = -5
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(t):
        return lib.cp_partial_attn_prefill(
            dev["q"], dev["cu_seqlens_q"], 2, mode=lib.CP_PASS_Q, k_cache=dev["k_cache"],
            v_cache=dev["v_cache"], block_tables=t.to(DEV), seq_lens_kv=dev["seq_lens"],
            interleave=8, impl=_impl_code(lib, impl), err=err, max_seqlen_q=20)

    run(tables)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    err.zero_()
    out, lse = run(x["block_tables"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], 2, 8, 16, 1 / 8)
    check_partials(out, lse, O, L, what=f"pass-Q {impl} after a bad table")


@pytest.mark.parametrize("impl", ["simt", "tc", "tc1"])
def test_pass_q_reports_short_kv(lib, impl):
    """seq_lens_kv below the new-query count (a negative cached context) lives on the device, so
    the kernels flag it (CP_ERR_DEVICE_BOUNDS) and skip the rows instead of running on."""
    x = _paged_case(2, [40, 30], [100, 60], 8, 2, 128, torch.bfloat16, 2, 8, 31)
    sl = torch.tensor([100, 20], dtype=torch.int32, device=DEV)   # sequence 1: 20 < 30
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.cp_partial_attn_prefill(x["q"].to(DEV), x["cu_seqlens_q"].to(DEV), 2, mode=lib.CP_PASS_Q,
                                k_cache=x["k_cache"].to(DEV), v_cache=x["v_cache"].to(DEV),
                                block_tables=x["block_tables"].to(DEV), seq_lens_kv=sl,
                                interleave=8, impl=_impl_code(lib, impl), err=err, max_seqlen_q=40)
    torch.cuda.synchronize()
    assert int(err.item()) == 5


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("case", [0, 1, 2, 4, 5, 6])
def test_fused_pass_q_parity(lib, case, split):
    """cp_attn_prefill_fused over the paged round-robin cache (every rank's resident pages in
    one online softmax) = merged pass-Q partials of the oracle; with the tail wave split into
    rank ranges (a workspace) and with every item whole (none)."""
    q_lens, kv_lens, Hq, Hkv, d, dt, cp, I = PASS_Q_CASES[case]
    x = _paged_case(len(q_lens), q_lens, kv_lens, Hq, Hkv, d, dt, cp, I, 300 + case)
    need = lib.cp_prefill_fused_workspace_size(len(q_lens), Hq, Hkv, d, cp, max(q_lens))
    if cp > 1 and case != 5:   # these grids leave most of their last wave's SMs idle
        assert need > 0
    ws = torch.empty(need if split else 0, dtype=torch.uint8, device=DEV)
    out, lse = lib.cp_attn_prefill_fused(
        x["q"].to(DEV), x["cu_seqlens_q"].to(DEV), cp, mode=lib.CP_PASS_Q,
        k_cache=x["k_cache"].to(DEV), v_cache=x["v_cache"].to(DEV),
        block_tables=x["block_tables"].to(DEV), seq_lens_kv=x["seq_lens"].to(DEV), interleave=I,
        max_seqlen_q=max(q_lens), workspace=ws)
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    check_merged(out, lse, Om, Lm, what=f"fused pass-Q split={split}")


@pytest.mark.parametrize("interleave", [(1 << 29) - 1, 1 << 30])
def test_pass_q_huge_interleave(lib, interleave):
    """An interleave size above every position deals all tokens to rank 0 (the others hold
    none): interleave x cp just below 2^31 and far above it, the two forms of the kernel's
    32-bit rank lengths.  Partials and the fused launch (with and without the tail split)."""
    q_lens, kv_lens, Hq, Hkv, d, cp = [300, 77], [900, 400], 8, 2, 128, 4
    g = torch.Generator().manual_seed(77)
    pages = [-(-L // 16) for L in kv_lens]
    pool = sum(pages)
    tables = torch.full((cp, len(q_lens), max(pages)), -1, dtype=torch.int32)
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    o = 0
    for b, n in enumerate(pages):  # rank 0 holds every token; the other ranks have no pages
        tables[0, b, :n] = perm[o:o + n]
        o += n
    q = wl.normal((sum(q_lens), Hq, d), torch.bfloat16, g)
    kc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g)
    vc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g)
    cu, sl = _cu(q_lens), torch.tensor(kv_lens, dtype=torch.int32)
    kw = dict(mode=lib.CP_PASS_Q, k_cache=kc.to(DEV), v_cache=vc.to(DEV), block_tables=tables.to(DEV),
              seq_lens_kv=sl.to(DEV), interleave=interleave, max_seqlen_q=max(q_lens))
    O, L = orc.pass_q_partials(q, kc, vc, tables, cu, sl, cp, interleave, 16, 1 / math.sqrt(d))
    assert np.isneginf(L[1:]).all()   # ranks 1.. hold nothing
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = lib.cp_partial_attn_prefill(q.to(DEV), cu.to(DEV), cp, err=err, **kw)
    check_partials(out, lse, O, L, what=f"pass-Q I={interleave}")
    Om, Lm = orc.lse_merge(O, L)
    for split in (True, False):
        need = lib.cp_prefill_fused_workspace_size(len(q_lens), Hq, Hkv, d, cp, max(q_lens))
        ws = torch.empty(need if split else 0, dtype=torch.uint8, device=DEV)
        fo, fl = lib.cp_attn_prefill_fused(q.to(DEV), cu.to(DEV), cp, workspace=ws, **kw)
        check_merged(fo, fl, Om, Lm, what=f"fused pass-Q I={interleave} split={split}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_max_cp(lib):
    """cp = 64, the largest the boundary accepts: 128 chunks per sequence (most a few tokens or
    empty), 64-rank walks, the fused pass-Q split plan over 64 ranks, and a fused decode at its
    limit of 256 partials (64 ranks x 4 splits)."""
    cp, d, bf = 64, 128, torch.bfloat16
    # pass-KV: partials (both tensor-core kernels) and the fused launch
    lens = [1000, 200, 3]
    x = wl.prefill_inputs(lens, 8, 2, d, bf, seed=640)
    # partials of 8-token chunks are dominated by a few keys: the outputs get the bound of the
    # probabilities' bf16 rounding, 2^-8 x the oracle's attention of |V|
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Oa, _ = orc.pass_kv_partials(x["q"], x["k"], x["v"].abs(), x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    Oam, _ = orc.lse_merge(Oa, L)
    args = (x["q"].to(DEV), x["cu_seqlens"].to(DEV), cp)
    for impl in (lib.CP_IMPL_TCGEN05, lib.CP_IMPL_TCGEN05_SINGLE):
        out, lse = lib.cp_partial_attn_prefill(*args, k=x["k"].to(DEV), v=x["v"].to(DEV),
                                               max_seqlen_q=max(lens), impl=impl)
        check_partials(out, lse, O, L, what=f"pass-KV cp=64 impl={impl}", o_abs=Oa)
    fo, fl = lib.cp_attn_prefill_fused(*args, x["k"].to(DEV), x["v"].to(DEV), max_seqlen_q=max(lens))
    check_merged(fo, fl, Om, Lm, what="fused pass-KV cp=64", o_abs=Oam)
    # pass-Q over a paged round-robin cache, interleave 4
    q_lens, kv_lens, I = [100, 40], [3000, 900], 4
    z = _paged_case(2, q_lens, kv_lens, 8, 2, d, bf, cp, I, 641)
    kw = dict(mode=lib.CP_PASS_Q, k_cache=z["k_cache"].to(DEV), v_cache=z["v_cache"].to(DEV),
              block_tables=z["block_tables"].to(DEV), seq_lens_kv=z["seq_lens"].to(DEV),
              interleave=I, max_seqlen_q=max(q_lens))
    Oq, Lq = orc.pass_q_partials(z["q"], z["k_cache"], z["v_cache"], z["block_tables"],
                                 z["cu_seqlens_q"], z["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Oqa, _ = orc.pass_q_partials(z["q"], z["k_cache"], z["v_cache"].abs(), z["block_tables"],
                                 z["cu_seqlens_q"], z["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    out, lse = lib.cp_partial_attn_prefill(z["q"].to(DEV), z["cu_seqlens_q"].to(DEV), cp, **kw)
    check_partials(out, lse, Oq, Lq, what="pass-Q cp=64", o_abs=Oqa)
    Oqm, Lqm = orc.lse_merge(Oq, Lq)
    Oqam, _ = orc.lse_merge(Oqa, Lq)
    need = lib.cp_prefill_fused_workspace_size(2, 8, 2, d, cp, max(q_lens))
    for ws in (torch.empty(need, dtype=torch.uint8, device=DEV),
               torch.empty(0, dtype=torch.uint8, device=DEV)):
        fo, fl = lib.cp_attn_prefill_fused(z["q"].to(DEV), z["cu_seqlens_q"].to(DEV), cp,
                                           workspace=ws, **kw)
        check_merged(fo, fl, Oqm, Lqm, what=f"fused pass-Q cp=64 workspace={ws.numel()}",
                     o_abs=Oqam)
    # decode: 64 ranks x 4 splits = 256 partials, the fused form's limit
    dl = [4000, 100, 1]
    y = wl.paged_inputs(3, 1, dl, 8, 2, d, bf, cp, 2, 16, 642, 643, q_is_decode=True)
    dev = {n: y[n].to(DEV) for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    ns, st = lib.cp_decode_plan(3, 2, cp, 2, 16, max(dl))
    assert cp * ns <= 256
    Od, Ld = orc.decode_partials(y["q"], y["k_cache"], y["v_cache"], y["block_tables"],
                                 y["seq_lens"], cp, 2, 16, 1 / math.sqrt(d))
    Odm, Ldm = orc.lse_merge(Od, Ld)
    Oda, _ = orc.decode_partials(y["q"], y["k_cache"], y["v_cache"].abs(), y["block_tables"],
                                 y["seq_lens"], cp, 2, 16, 1 / math.sqrt(d))
    Odam, _ = orc.lse_merge(Oda, Ld)
    po, pl = lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_tables"], dev["seq_lens"], cp, 2,
                                        num_splits=ns, split_tokens=st)
    mo, ml = lib.cp_lse_merge(po, pl, out_dtype=bf)
    check_merged(mo, ml, Odm, Ldm, what="decode cp=64", o_abs=Odam)
    fd, fdl = lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                      dev["block_tables"], dev["seq_lens"], cp, 2,
                                      num_splits=ns, split_tokens=st)
    check_merged(fd, fdl, Odm, Ldm, what="fused decode cp=64", o_abs=Odam)


def test_many_short_sequences(lib):
    """300 sequences of 1-40 tokens (most chunks a token or two, many empty): the work-item
    decode over a long sequence index, pass-KV and pass-Q, partials and fused."""
    g = torch.Generator().manual_seed(650)
    lens = (torch.randint(1, 41, (300,), generator=g)).tolist()
    cp, d, bf = 3, 128, torch.bfloat16
    x = wl.prefill_inputs(lens, 8, 2, d, bf, seed=651)
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Oa, _ = orc.pass_kv_partials(x["q"], x["k"], x["v"].abs(), x["cu_seqlens"], cp, 1 / math.sqrt(d))
    args = (x["q"].to(DEV), x["cu_seqlens"].to(DEV), cp)
    out, lse = lib.cp_partial_attn_prefill(*args, k=x["k"].to(DEV), v=x["v"].to(DEV),
                                           max_seqlen_q=max(lens))
    check_partials(out, lse, O, L, what="pass-KV 300 sequences", o_abs=Oa)
    Om, Lm = orc.lse_merge(O, L)
    Oam, _ = orc.lse_merge(Oa, L)
    fo, fl = lib.cp_attn_prefill_fused(*args, x["k"].to(DEV), x["v"].to(DEV), max_seqlen_q=max(lens))
    check_merged(fo, fl, Om, Lm, what="fused pass-KV 300 sequences", o_abs=Oam)
    # the same new tokens as chunks of longer paged sequences (pass-Q)
    kv_lens = [n + int(c) for n, c in zip(lens, torch.randint(0, 200, (300,), generator=g))]
    z = _paged_case(300, lens, kv_lens, 8, 2, d, bf, cp, 8, 652)
    kw = dict(mode=lib.CP_PASS_Q, k_cache=z["k_cache"].to(DEV), v_cache=z["v_cache"].to(DEV),
              block_tables=z["block_tables"].to(DEV), seq_lens_kv=z["seq_lens"].to(DEV),
              interleave=8, max_seqlen_q=max(lens))
    Oq, Lq = orc.pass_q_partials(z["q"], z["k_cache"], z["v_cache"], z["block_tables"],
                                 z["cu_seqlens_q"], z["seq_lens"], cp, 8, 16, 1 / math.sqrt(d))
    Oqa, _ = orc.pass_q_partials(z["q"], z["k_cache"], z["v_cache"].abs(), z["block_tables"],
                                 z["cu_seqlens_q"], z["seq_lens"], cp, 8, 16, 1 / math.sqrt(d))
    out, lse = lib.cp_partial_attn_prefill(z["q"].to(DEV), z["cu_seqlens_q"].to(DEV), cp, **kw)
    check_partials(out, lse, Oq, Lq, what="pass-Q 300 sequences", o_abs=Oqa)
    Oqm, Lqm = orc.lse_merge(Oq, Lq)
    Oqam, _ = orc.lse_merge(Oqa, Lq)
    fo, fl = lib.cp_attn_prefill_fused(z["q"].to(DEV), z["cu_seqlens_q"].to(DEV), cp, **kw)
    check_merged(fo, fl, Oqm, Lqm, what="fused pass-Q 300 sequences", o_abs=Oqam)


# ------------------------------------------------------------------------------------ decode

DECODE_CASES = [
    # B, lens range, Hq, Hkv, d, dtype, cp, I
    (5, (1, 3000), 32, 8, 128, torch.bfloat16, 2, 8),
    (3, (1, 40), 16, 2, 64, torch.bfloat16, 4, 8),
    (7, (500, 900), 8, 8, 128, torch.float32, 3, 4),
    (2, (1000, 2000), 16, 16, 64, torch.bfloat16, 1, 8),
    (4, (100, 2500), 28, 4, 128, torch.bfloat16, 2, 8),   # G = 7
    (3, (50, 700), 15, 5, 64, torch.bfloat16, 3, 16),     # G = 3
    (2, (200, 900), 10, 2, 128, torch.float32, 2, 8),     # G = 5, CUDA-core kernel
    (3, (100, 1500), 32, 2, 128, torch.bfloat16, 2, 8),   # G = 16: both MMA row halves
    (2, (30, 600), 11, 1, 64, torch.bfloat16, 3, 4),      # G = 11
]


@pytest.mark.parametrize("case", range(len(DECODE_CASES)))
def test_decode_parity(lib, case):
    B, (lo, hi), Hq, Hkv, d, dt, cp, I = DECODE_CASES[case]
    lens = wl.decode_lengths(B, lo, hi, seed=400 + case).tolist()
    lens[0] = hi                                   # longest sequence present
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, dt, cp, I, 16, 500 + case, 600 + case,
                        q_is_decode=True)
    out, lse = lib.cp_partial_attn_decode(
        x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV), x["block_tables"].to(DEV),
        x["seq_lens"].to(DEV), cp, I, max_seq_len=max(lens))
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"], x["seq_lens"],
                               cp, I, 16, 1 / math.sqrt(d))
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=dt)
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what="decode merged")
    # per-rank partials: merge the GPU's splits of each rank and compare with the oracle's rank
    S = out.shape[0] // cp
    for r in range(cp):
        ro, rl = lib.cp_lse_merge(out[r * S:(r + 1) * S].contiguous(),
                                  lse[r * S:(r + 1) * S].contiguous(), out_dtype=torch.float32)
        check_partials(ro[None], rl[None], O[r:r + 1], L[r:r + 1], what=f"decode rank {r}")


def test_decode_explicit_single_split(lib):
    """One split per rank: the decode partials are exactly the per-rank partials."""
    B, Hq, Hkv, d, cp, I = 3, 16, 4, 128, 2, 8
    lens = [33, 1, 250]
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, 11, 12, q_is_decode=True)
    out, lse = lib.cp_partial_attn_decode(
        x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV), x["block_tables"].to(DEV),
        x["seq_lens"].to(DEV), cp, I, num_splits=1, split_tokens=128)
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"], x["seq_lens"],
                               cp, I, 16, 1 / math.sqrt(d))
    check_partials(out, lse, O, L, what="decode single split")


@pytest.mark.parametrize("case", range(len(DECODE_CASES)))
def test_decode_fused_parity(lib, case):
    """cp_decode_attention (partials + merge in one launch) against the oracle, twice on the
    same workspace (its arrival counters must come back to zero), and against the two-launch
    path."""
    B, (lo, hi), Hq, Hkv, d, dt, cp, I = DECODE_CASES[case]
    lens = wl.decode_lengths(B, lo, hi, seed=400 + case).tolist()
    lens[0] = hi
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, dt, cp, I, 16, 500 + case, 600 + case,
                        q_is_decode=True)
    dev = {n: x[n].to(DEV) for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    ns, st = lib.cp_decode_plan(B, Hkv, cp, I, 16, max(lens))
    ws = torch.zeros(lib.cp_decode_workspace_size(B, Hq, Hkv, d, cp, ns), dtype=torch.uint8,
                     device=DEV)
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"], x["seq_lens"],
                               cp, I, 16, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    outs = []
    for _ in range(2):
        out, lse = lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                           dev["block_tables"], dev["seq_lens"], cp, I,
                                           num_splits=ns, split_tokens=st, workspace=ws)
        check_merged(out, lse, Om, Lm, what="fused decode")
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])
    counters = ws[: B * Hkv * 4].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0
    po, pl = lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_tables"], dev["seq_lens"], cp, I,
                                        num_splits=ns, split_tokens=st)
    mo, _ = lib.cp_lse_merge(po, pl, out_dtype=dt)
    check_same_rounded(outs[0], mo, what="fused decode vs partials + merge")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_decode_reports_bad_page(lib, dt):
    """Decode (tensor-core bf16 and CUDA-core f32 kernels) checks every visible page id: an entry
    outside the pool is skipped and flagged, and the next valid call still matches."""
    B, Hq, Hkv, d, cp, I = 2, 16, 4, 128, 2, 8
    lens = [700, 300]
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, dt, cp, I, 16, 21, 22, q_is_decode=True)
    dev = {n: x[n].to(DEV) for n in ("q", "k_cache", "v_cache", "seq_lens")}
    tables = x["block_tables"].clone()
    tables[0, 0, 2] = 10 ** 6
    tables[1, 1, 0] = -1
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(t):
        return lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"], t.to(DEV),
                                          dev["seq_lens"], cp, I, max_seq_len=max(lens), err=err)

    run(tables)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    err.zero_()
    out, lse = run(x["block_tables"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    mo, ml = lib.cp_lse_merge(out, lse, out_dtype=dt)
    Om, Lm = orc.lse_merge(O, L)
    check_merged(mo, ml, Om, Lm, what="decode after a bad table")


def test_decode_fused_rejects_small_workspace(lib):
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(1, 4, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros(1, 2, 2, dtype=torch.int32, device=DEV)
    lens = torch.tensor([3, 5], dtype=torch.int32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.CPError) as e:
        lib.cp_decode_attention(q, kc, kc, tables, lens, 1, 8, num_splits=1, split_tokens=16,
                                workspace=ws)
    assert e.value.status == 1 and "workspace" in e.value.detail


# ------------------------------------------------------------------------------------ cache write

@pytest.mark.parametrize("dt,d,cp,I", [(torch.bfloat16, 128, 2, 8), (torch.float32, 64, 3, 4),
                                       (torch.bfloat16, 64, 4, 1)])
def test_kv_cache_write_bitexact(lib, dt, d, cp, I):
    """New tokens written at their round-robin slots: every byte of the pools equals the oracle's
    placement (untouched slots keep their old values)."""
    g = torch.Generator().manual_seed(77 + cp)
    Hkv, bs = 4, 16
    cached = [100, 0, 37]
    new = [5, 64, 1]
    caps = [wl.block_capacity(c + n, cp, I, bs) for c, n in zip(cached, new)]
    tables, pool = wl.shuffled_block_tables(caps, cp, g)
    kc = wl.normal((cp, pool, Hkv, bs, d), dt, g)
    vc = wl.normal((cp, pool, Hkv, bs, d), dt, g)
    kn = wl.normal((sum(new), Hkv, d), dt, g)
    vn = wl.normal((sum(new), Hkv, d), dt, g)
    cu = _cu(new)
    start = torch.tensor(cached, dtype=torch.int32)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lib.cp_kv_cache_write(kn.to(DEV), vn.to(DEV), cu.to(DEV), start.to(DEV), kd, vd,
                          tables.to(DEV), cp, I)
    kr, vr = kc.clone(), vc.clone()
    orc.kv_cache_write(kn, vn, cu, start, cp, I, bs, tables, kr, vr)
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)


def test_kv_cache_write_reports_missing_page(lib):
    tables = torch.full((2, 1, 1), 0, dtype=torch.int32)     # one page: 16 local tokens per rank
    kc = torch.zeros(2, 1, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    kn = torch.ones(40, 1, 64, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.cp_kv_cache_write(kn, kn, _cu([40]).to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
                          kc, kc.clone(), tables.to(DEV), 2, 8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    assert int((kc != 0).any(dim=-1).sum().item()) == 32    # 16 slots per rank written


# ------------------------------------------------------------------------------------ fused prefill

@pytest.mark.parametrize("case", [1, 2, 3, 4, 6, 7])
def test_fused_prefill_parity(lib, case):
    """cp_attn_prefill_fused = merged pass-KV partials = plain causal attention."""
    lens, Hq, Hkv, d, dt, cp = PASS_KV_CASES[case]
    x = wl.prefill_inputs(lens, Hq, Hkv, d, dt, seed=100 + case)
    out, lse = lib.cp_attn_prefill_fused(x["q"].to(DEV), x["cu_seqlens"].to(DEV), cp,
                                         x["k"].to(DEV), x["v"].to(DEV), max_seqlen_q=max(lens))
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    check_merged(out, lse, Om, Lm, what="fused prefill")
