"""Hot paths captured in a CUDA graph and replayed: same results (bitwise) as the eager calls,
over several replays, and the replayed results equal the float64 oracle within the parity
tolerances (so a fault shared by the eager and the captured call, such as a stale tensor map,
cannot pass).  The pages turn prefill CP off under full CUDA graphs ("[Feature] Prefill Context
Parallel (PCP) basic support", code-review summary); here the prefill path (partition ->
partials -> merge, or the fused launch) and the decode path (layout -> split partials -> merge,
or the fused launch with its self-resetting counters) are capturable: every call is
stream-ordered and allocates nothing when its outputs are given."""
import math

import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_merged

pytestmark = pytest.mark.gpu


def _capture_and_replay(step, outs):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # eager warm-up (attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    refs = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o, r)


def _decode_setup(lib):
    B, Hq, Hkv, d, cp, I = 6, 32, 8, 128, 2, 8
    lens = wl.decode_lengths(B, 100, 5000, seed=71).tolist()
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, 72, 73, q_is_decode=True)
    dev = {n: x[n].cuda() for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    cu = torch.tensor([0] + torch.tensor(lens).cumsum(0).tolist(), dtype=torch.int32, device="cuda")
    ns, st = lib.cp_decode_plan(B, Hkv, cp, I, 16, max(lens))
    return B, Hq, Hkv, d, cp, I, lens, dev, cu, ns, st, x


def _decode_oracle(x, lens, cp, I, d):
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    return orc.lse_merge(O, L)


def test_decode_path_in_a_cuda_graph(lib):
    B, Hq, Hkv, d, cp, I, lens, dev, cu, ns, st, x = _decode_setup(lib)
    part = torch.empty(cp * ns, B, Hq, d, device="cuda")
    plse = torch.empty(cp * ns, B, Hq, device="cuda")
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")
    ll = torch.empty(cp, B, dtype=torch.int32, device="cuda")

    def step():
        lib.cp_kv_interleave_layout(cu, cp, I, 0, 16, local_lens=ll, want_slots=False)
        lib.cp_partial_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], cp, I, num_splits=ns, split_tokens=st,
                                   out=part, lse=plse)
        lib.cp_lse_merge(part, plse, out=out, out_lse=lse)

    _capture_and_replay(step, [out, lse])
    Om, Lm = _decode_oracle(x, lens, cp, I, d)
    check_merged(out, lse, Om, Lm, "decode graph replay")


def test_fused_decode_in_a_cuda_graph(lib):
    """The arrival counters in the workspace return to zero after every launch, so the same
    captured launch replays correctly."""
    B, Hq, Hkv, d, cp, I, lens, dev, cu, ns, st, x = _decode_setup(lib)
    ws = torch.zeros(lib.cp_decode_workspace_size(B, Hq, Hkv, d, cp, ns), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")

    def step():
        lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                dev["seq_lens"], cp, I, num_splits=ns, split_tokens=st,
                                workspace=ws, out=out, out_lse=lse)

    _capture_and_replay(step, [out, lse])
    Om, Lm = _decode_oracle(x, lens, cp, I, d)
    check_merged(out, lse, Om, Lm, "fused decode graph replay")


@pytest.mark.parametrize("fused", [False, True])
def test_prefill_path_in_a_cuda_graph(lib, fused):
    lens, Hq, Hkv, d, cp = [1000, 2300], 8, 2, 128, 2
    x = wl.prefill_inputs(lens, Hq, Hkv, d, torch.bfloat16, seed=74)
    q, k, v, cu = (x[n].cuda() for n in ("q", "k", "v", "cu_seqlens"))
    N = sum(lens)
    perm = torch.empty(N, dtype=torch.int32, device="cuda")
    inv = torch.empty(N, dtype=torch.int32, device="cuda")
    so = torch.empty(cp + 1, dtype=torch.int32, device="cuda")
    cb = torch.empty(len(lens), 2 * cp + 1, dtype=torch.int32, device="cuda")
    part = torch.empty(cp, N, Hq, d, device="cuda")
    plse = torch.empty(cp, N, Hq, device="cuda")
    out = torch.empty(N, Hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(N, Hq, device="cuda")

    def step():
        lib.cp_partition(cu, cp, N, perm, inv, so, cb)
        if fused:
            lib.cp_attn_prefill_fused(q, cu, cp, k, v, max_seqlen_q=max(lens), out=out,
                                      out_lse=lse)
        else:
            lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=max(lens), out=part,
                                        lse=plse)
            lib.cp_lse_merge(part, plse, out=out, out_lse=lse)

    _capture_and_replay(step, [out, lse, perm])
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    check_merged(out, lse, Om, Lm, f"prefill graph replay (fused={fused})")
    assert perm.cpu().numpy().tolist() == orc.partition(lens, cp)["perm"].tolist()


@pytest.mark.parametrize("fused", [False, True])
def test_pass_q_path_in_a_cuda_graph(lib, fused):
    """Chunked prefill over the paged round-robin cache (pass-Q): partials + merge, or the fused
    launch that walks every rank's pages."""
    B, q_len, kv_lens, Hq, Hkv, d, cp, I = 2, 300, [1500, 900], 8, 2, 128, 2, 8
    x = wl.paged_inputs(B, q_len, kv_lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, 75, 76)
    dev = {n: x[n].cuda() for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens",
                                    "cu_seqlens_q")}
    N = B * q_len
    part = torch.empty(cp, N, Hq, d, device="cuda")
    plse = torch.empty(cp, N, Hq, device="cuda")
    out = torch.empty(N, Hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(N, Hq, device="cuda")
    kw = dict(mode=lib.CP_PASS_Q, k_cache=dev["k_cache"], v_cache=dev["v_cache"],
              block_tables=dev["block_tables"], seq_lens_kv=dev["seq_lens"], interleave=I,
              max_seqlen_q=q_len)

    # 32 equal items on 152 SMs: the fused launch splits them by rank range (+ a merge kernel)
    ws = torch.empty(lib.cp_prefill_fused_workspace_size(B, Hq, Hkv, d, cp, q_len),
                     dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0

    def step():
        if fused:
            lib.cp_attn_prefill_fused(dev["q"], dev["cu_seqlens_q"], cp, out=out, out_lse=lse,
                                      workspace=ws, **kw)
        else:
            lib.cp_partial_attn_prefill(dev["q"], dev["cu_seqlens_q"], cp, out=part, lse=plse, **kw)
            lib.cp_lse_merge(part, plse, out=out, out_lse=lse)

    _capture_and_replay(step, [out, lse])
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    check_merged(out, lse, Om, Lm, f"pass-Q graph replay (fused={fused})")
