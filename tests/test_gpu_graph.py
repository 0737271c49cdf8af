"""The decode path (layout -> per-rank split partials -> merge) captured in a CUDA graph and
replayed: same results as the eager calls, over several replays (the pages disable prefill CP
under full CUDA graphs; this library's decode path is capturable)."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def test_decode_path_in_a_cuda_graph(lib):
    B, Hq, Hkv, d, cp, I = 6, 32, 8, 128, 2, 8
    lens = wl.decode_lengths(B, 100, 5000, seed=71).tolist()
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, 72, 73, q_is_decode=True)
    dev = {n: x[n].cuda() for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    cu = torch.tensor([0] + torch.tensor(lens).cumsum(0).tolist(), dtype=torch.int32, device="cuda")
    ns, st = lib.cp_decode_plan(B, Hkv, cp, I, 16, max(lens))
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

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # eager warm-up (attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref, ref_lse = out.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
