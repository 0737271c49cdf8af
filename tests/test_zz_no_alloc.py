"""cp_decode_attention_noalloc: the decode entry point for callers that cannot allocate device
memory when they call it (a framework that owns the whole memory pool, a fixed-footprint
serving process).  It must give the same result as cp_decode_attention, which takes a caller-
allocated workspace, and keep doing so on consecutive calls that share its built-in scratch;
each call's output is also checked against the float64 oracle (decode partials + LSE merge).

Collected last on purpose; it passes alone in a fresh process and after the other tests.
"""
import ctypes
import math

import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_merged

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(seed):
    B, Hq, Hkv, d, cp, I = 8, 32, 8, 128, 2, 8
    lens = wl.decode_lengths(B, 1, 6000, seed=seed).tolist()
    lens[0] = 6000
    x = wl.paged_inputs(B, 1, lens, Hq, Hkv, d, torch.bfloat16, cp, I, 16, seed + 1, seed + 2,
                        q_is_decode=True)
    dev = {n: x[n].to(DEV) for n in ("q", "k_cache", "v_cache", "block_tables", "seq_lens")}
    return dev, B, Hq, Hkv, d, cp, I, max(lens), x


def test_noalloc_matches_workspace_entry_point_twice(lib):
    dev, B, Hq, Hkv, d, cp, I, maxlen, x = _case(901)
    O, L = orc.decode_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], cp, I, 16, 1 / math.sqrt(d))
    Om, Lm = orc.lse_merge(O, L)
    ns, st = lib.cp_decode_plan(B, Hkv, cp, I, 16, maxlen)
    assert lib.cp_decode_workspace_size(B, Hq, Hkv, d, cp, ns) <= lib.NOALLOC_SCRATCH_BYTES
    ref, ref_lse = lib.cp_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                           dev["block_tables"], dev["seq_lens"], cp, I,
                                           num_splits=ns, split_tokens=st)
    for call in range(2):  # the second call reuses whatever the first left in the scratch
        out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
        lib.cp_decode_attention_noalloc(dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_tables"], dev["seq_lens"], cp, I, out,
                                        num_splits=ns, split_tokens=st, out_lse=lse)
        torch.cuda.synchronize()
        assert (out.float() - ref.float()).abs().max().item() <= 1e-2, call
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        assert ((lse[fin] - ref_lse[fin]).abs() <= 1e-3 * ref_lse[fin].abs() + 1e-5).all(), call
        check_merged(out, lse, Om, Lm, f"no-alloc decode, call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # 64 sequences x 32 heads x 128 floats per partial = 1 MiB; 2 ranks x 32 splits = 64 MiB.
    # The host rejects the size before anything is launched.
    B, Hq, Hkv, d, cp, I, ns = 64, 32, 8, 128, 2, 8, 32
    assert lib.cp_decode_workspace_size(B, Hq, Hkv, d, cp, ns) > lib.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(cp, 1, Hkv, 16, d, dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros(cp, B, 1, dtype=torch.int32, device=DEV)
    lens = torch.ones(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(lib.CPError) as e:
        lib.cp_decode_attention_noalloc(q, kc, kc, tables, lens, cp, I, out, num_splits=ns,
                                        split_tokens=16)
    assert e.value.status == 1 and "scratch" in e.value.detail


def test_noalloc_is_exported_through_the_c_abi(lib):
    raw = ctypes.CDLL(lib.lib_path())
    assert hasattr(raw, "cp_decode_attention_noalloc")
