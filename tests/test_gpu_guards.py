"""Guard regions around every output buffer (the stand-in for a memory checker, which is not
available on this pool): each output is a view into a larger buffer whose leading and trailing
words hold a canary bit pattern; after the call the canaries must be intact bit for bit, so no
kernel wrote outside the rows, heads and pages it was given.  Shapes are ragged on purpose
(partial tiles, empty ranks, short contexts)."""
import math

import pytest
import torch

import workloads as wl
from tests.parity_util import check_same_rounded

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 64          # elements on each side; keeps the view 128-byte aligned for bf16 and f32
CANARY = {torch.float32: 0x7FC0DEAD, torch.bfloat16: 0x7FAD, torch.int32: 0x5A5A5A5A}


def _guarded(shape, dtype):
    n = math.prod(shape)
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=DEV)
    ibuf = buf.view(torch.int32 if dtype != torch.bfloat16 else torch.int16)
    ibuf.fill_(CANARY[dtype] if dtype != torch.bfloat16 else CANARY[dtype])
    view = buf[GUARD:GUARD + n].view(shape)
    return buf, view


def _intact(buf, dtype, what):
    ibuf = buf.view(torch.int32 if dtype != torch.bfloat16 else torch.int16)
    want = CANARY[dtype]
    head, tail = ibuf[:GUARD].cpu(), ibuf[-GUARD:].cpu()
    assert bool((head == want).all()) and bool((tail == want).all()), f"{what}: guard overwritten"


@pytest.mark.parametrize("lens,Hq,Hkv,d,cp", [([700, 129, 1], 8, 2, 128, 2), ([333], 8, 2, 64, 3),
                                             ([90], 4, 1, 128, 4)])
def test_prefill_partials_merge_and_fused_stay_in_bounds(lib, lens, Hq, Hkv, d, cp):
    x = wl.prefill_inputs(lens, Hq, Hkv, d, torch.bfloat16, seed=91)
    q, k, v, cu = (x[n].to(DEV) for n in ("q", "k", "v", "cu_seqlens"))
    N = sum(lens)
    pb, part = _guarded((cp, N, Hq, d), torch.float32)
    lb, plse = _guarded((cp, N, Hq), torch.float32)
    lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=max(lens), out=part, lse=plse)
    ob, out = _guarded((N, Hq, d), torch.bfloat16)
    olb, olse = _guarded((N, Hq), torch.float32)
    lib.cp_lse_merge(part, plse, out=out, out_lse=olse)
    fb, fout = _guarded((N, Hq, d), torch.bfloat16)
    flb, flse = _guarded((N, Hq), torch.float32)
    lib.cp_attn_prefill_fused(q, cu, cp, k, v, max_seqlen_q=max(lens), out=fout, out_lse=flse)
    torch.cuda.synchronize()
    for b, dt, w in ((pb, torch.float32, "partials"), (lb, torch.float32, "partial lse"),
                     (ob, torch.bfloat16, "merged out"), (olb, torch.float32, "merged lse"),
                     (fb, torch.bfloat16, "fused out"), (flb, torch.float32, "fused lse")):
        _intact(b, dt, w)
    check_same_rounded(fout, out, what="fused vs partials + merge")


def test_pass_q_and_decode_stay_in_bounds(lib):
    B, Hq, Hkv, d, cp, I = 3, 8, 2, 128, 4, 8
    q_lens, kv_lens = [100, 1, 37], [700, 17, 300]
    g = torch.Generator().manual_seed(92)
    caps = [wl.block_capacity(L, cp, I, 16) for L in kv_lens]
    tables, pool = wl.shuffled_block_tables(caps, cp, g)
    kc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g).to(DEV)
    vc = wl.normal((cp, pool, Hkv, 16, d), torch.bfloat16, g).to(DEV)
    q = wl.normal((sum(q_lens), Hq, d), torch.bfloat16, g).to(DEV)
    cu_q = torch.tensor([0, 100, 101, 138], dtype=torch.int32, device=DEV)
    sl = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    td = tables.to(DEV)
    N = sum(q_lens)
    pb, part = _guarded((cp, N, Hq, d), torch.float32)
    lb, plse = _guarded((cp, N, Hq), torch.float32)
    lib.cp_partial_attn_prefill(q, cu_q, cp, mode=lib.CP_PASS_Q, k_cache=kc, v_cache=vc,
                                block_tables=td, seq_lens_kv=sl, interleave=I, max_seqlen_q=100,
                                out=part, lse=plse)
    qd = wl.normal((B, Hq, d), torch.bfloat16, g).to(DEV)
    ns, st = lib.cp_decode_plan(B, Hkv, cp, I, 16, max(kv_lens))
    db, dpart = _guarded((cp * ns, B, Hq, d), torch.float32)
    dlb, dlse = _guarded((cp * ns, B, Hq), torch.float32)
    lib.cp_partial_attn_decode(qd, kc, vc, td, sl, cp, I, num_splits=ns, split_tokens=st,
                               out=dpart, lse=dlse)
    ws = torch.zeros(lib.cp_decode_workspace_size(B, Hq, Hkv, d, cp, ns), dtype=torch.uint8,
                     device=DEV)
    fb, fout = _guarded((B, Hq, d), torch.bfloat16)
    flb, flse = _guarded((B, Hq), torch.float32)
    lib.cp_decode_attention(qd, kc, vc, td, sl, cp, I, num_splits=ns, split_tokens=st,
                            workspace=ws, out=fout, out_lse=flse)
    torch.cuda.synchronize()
    for b, dt, w in ((pb, torch.float32, "pass-Q partials"), (lb, torch.float32, "pass-Q lse"),
                     (db, torch.float32, "decode partials"), (dlb, torch.float32, "decode lse"),
                     (fb, torch.bfloat16, "fused decode out"), (flb, torch.float32, "fused lse")):
        _intact(b, dt, w)


def test_kv_cache_write_stays_in_pages(lib):
    cp, I, Hkv, d = 2, 8, 2, 128
    g = torch.Generator().manual_seed(93)
    cached, new = [40, 0], [9, 33]
    caps = [wl.block_capacity(c + n, cp, I, 16) for c, n in zip(cached, new)]
    tables, pool = wl.shuffled_block_tables(caps, cp, g)
    kb, kc = _guarded((cp, pool, Hkv, 16, d), torch.bfloat16)
    vb, vc = _guarded((cp, pool, Hkv, 16, d), torch.bfloat16)
    kn = wl.normal((sum(new), Hkv, d), torch.bfloat16, g).to(DEV)
    vn = wl.normal((sum(new), Hkv, d), torch.bfloat16, g).to(DEV)
    cu = torch.tensor([0, 9, 42], dtype=torch.int32, device=DEV)
    start = torch.tensor(cached, dtype=torch.int32, device=DEV)
    lib.cp_kv_cache_write(kn, vn, cu, start, kc, vc, tables.to(DEV), cp, I)
    torch.cuda.synchronize()
    _intact(kb, torch.bfloat16, "k cache")
    _intact(vb, torch.bfloat16, "v cache")
