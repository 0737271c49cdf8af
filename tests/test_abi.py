"""The C ABI library loads on a machine without a GPU and exports every function that
include/*.h declares; host-side validation rejects bad arguments before any launch."""
import ctypes
import glob
import os
import re

import pytest

import context_gqa_attention_gb300 as cpa
from context_gqa_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(cp_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return cpa.load()


def test_header_declares_the_boundary():
    want = {"cp_partition", "cp_kv_interleave_layout", "cp_partial_attn_prefill",
            "cp_partial_attn_decode", "cp_lse_merge", "cp_decode_plan"}
    assert want <= _declared()


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(_build.LIB)
    for name in sorted(_declared()):
        assert hasattr(raw, name), name
    assert set(cpa.EXPORTED) <= _declared()


def test_struct_mirrors_match(lib):
    assert lib.cp_prefill_args_size() == ctypes.sizeof(cpa.PrefillArgs)
    assert lib.cp_decode_args_size() == ctypes.sizeof(cpa.DecodeArgs)
    assert lib.cp_abi_version() == 3
    assert lib.cp_status_string(5) == b"CP_ERR_DEVICE_BOUNDS"


def _last(lib):
    buf = ctypes.create_string_buffer(256)
    st = lib.cp_last_error(buf, 256)
    return st, buf.value.decode()


def test_invalid_arguments_are_rejected_on_the_host(lib):
    # null / bad pointers and sizes return an error without touching the device
    assert lib.cp_partition(None, 1, 10, 2, None, None, None, None, None) == 1
    assert "cu_seqlens" in _last(lib)[1]
    assert lib.cp_partition(ctypes.c_void_p(16), 1, 10, 0, ctypes.c_void_p(16), None, None, None,
                            None) == 1
    assert lib.cp_lse_merge(ctypes.c_void_p(16), ctypes.c_void_p(16), 2, 4, 2, 96,
                            ctypes.c_void_p(16), 1, None, None) == 1
    assert lib.cp_lse_merge(ctypes.c_void_p(18), ctypes.c_void_p(16), 2, 4, 2, 128,
                            ctypes.c_void_p(16), 1, None, None) == 1   # misaligned
    a = cpa.PrefillArgs()
    a.mode, a.dtype, a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.cp = 0, 1, 1, 6, 4, 128, 2
    assert lib.cp_partial_attn_prefill(ctypes.byref(a), None) == 1      # Hq % Hkv != 0
    assert "multiple" in _last(lib)[1]
    a.num_q_heads, a.head_dim = 8, 96
    assert lib.cp_partial_attn_prefill(ctypes.byref(a), None) == 2      # unsupported head_dim
    d = cpa.DecodeArgs()
    d.dtype, d.num_seqs, d.num_q_heads, d.num_kv_heads, d.head_dim = 1, 1, 32, 8, 128
    d.cp, d.interleave, d.block_size, d.num_splits, d.split_tokens = 2, 8, 32, 1, 64
    assert lib.cp_partial_attn_decode(ctypes.byref(d), None) == 2       # block size 32
    d.block_size, d.split_tokens = 16, 40
    assert lib.cp_partial_attn_decode(ctypes.byref(d), None) == 1       # split not page multiple


def test_fused_prefill_arguments_are_checked_on_the_host(lib):
    """cp_attn_prefill_fused: the pass-Q form needs the paged-cache arguments and the two-tile
    kernel; bad modes, f32 inputs and a misaligned workspace are refused before any launch."""
    fake = ctypes.c_void_p(256)

    def fused(f, out_lse=fake, ws=None, ws_bytes=0):
        return lib.cp_attn_prefill_fused(ctypes.byref(f), ws, ws_bytes, fake, out_lse, None)

    f = cpa.PrefillArgs()
    f.mode, f.dtype, f.num_seqs, f.num_q_heads, f.num_kv_heads, f.head_dim, f.cp = 1, 1, 1, 8, 2, 128, 2
    f.total_q, f.max_seqlen_q, f.q_shard, f.kv_shard = 10, 10, -1, -1
    f.cu_seqlens_q, f.q, f.k_cache, f.v_cache = 256, 256, 256, 256
    f.impl = cpa.CP_IMPL_TCGEN05_SINGLE
    assert fused(f) == 2
    assert "two-tile" in _last(lib)[1]
    f.impl = cpa.CP_IMPL_AUTO
    assert fused(f) == 1   # no block tables
    assert "block_tables" in _last(lib)[1]
    f.block_tables, f.seq_lens_kv, f.max_blocks, f.pool_pages, f.interleave = 256, 256, 4, 8, 8
    f.block_size = 32
    assert fused(f) == 2   # block size 32
    f.block_size = 16
    assert fused(f, out_lse=None) == 1   # no out_lse
    assert fused(f, ws=ctypes.c_void_p(256 + 16), ws_bytes=1 << 20) == 1   # misaligned workspace
    assert "workspace" in _last(lib)[1]
    f.mode = 7
    assert fused(f) == 1
    f.mode, f.dtype = 0, 0
    assert fused(f) == 2   # f32 inputs


def test_fused_prefill_workspace_size_on_the_host(lib):
    """cp_prefill_fused_workspace_size: shape checks, and no split (0 bytes) for pass-KV."""
    n = ctypes.c_size_t(123)
    f = cpa.PrefillArgs()
    f.mode, f.dtype, f.num_seqs, f.num_q_heads, f.num_kv_heads, f.head_dim, f.cp = 0, 1, 4, 16, 2, 128, 4
    f.total_q, f.max_seqlen_q, f.q_shard, f.kv_shard = 8192, 2048, -1, -1
    assert lib.cp_prefill_fused_workspace_size(ctypes.byref(f), ctypes.byref(n)) == 0
    assert n.value == 0
    assert lib.cp_prefill_fused_workspace_size(ctypes.byref(f), None) == 1
    f.head_dim = 96
    assert lib.cp_prefill_fused_workspace_size(ctypes.byref(f), ctypes.byref(n)) == 2
    f.head_dim, f.cp = 128, 0
    assert lib.cp_prefill_fused_workspace_size(ctypes.byref(f), ctypes.byref(n)) == 1
    f.cp, f.kv_shard = 4, 1
    assert lib.cp_prefill_fused_workspace_size(ctypes.byref(f), ctypes.byref(n)) == 1


def test_cached_context_arguments_are_checked_on_the_host(lib):
    """PASS_KV with cu_seqlens_kv needs kv rows when there are queries; PASS_Q refuses the
    PASS_KV-only kv lengths."""
    a = cpa.PrefillArgs()
    a.mode, a.dtype, a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.cp = 0, 1, 1, 8, 2, 128, 2
    a.total_q, a.max_seqlen_q, a.q_shard, a.kv_shard = 10, 10, -1, -1
    a.cu_seqlens_q, a.q, a.k, a.v, a.out, a.lse = 256, 256, 256, 256, 256, 256
    a.cu_seqlens_kv, a.total_kv = 256, 0
    assert lib.cp_partial_attn_prefill(ctypes.byref(a), None) == 1
    assert "total_kv" in _last(lib)[1]
    a.total_kv = -3
    assert lib.cp_partial_attn_prefill(ctypes.byref(a), None) == 1
    a.mode, a.k_cache, a.v_cache, a.block_tables, a.seq_lens_kv = 1, 256, 256, 256, 256
    a.max_blocks, a.pool_pages, a.interleave, a.block_size = 4, 8, 8, 16
    assert lib.cp_partial_attn_prefill(ctypes.byref(a), None) == 1
    assert "cu_seqlens_kv" in _last(lib)[1]


def test_decode_plan_covers_every_rank_share(lib):
    for B, Hkv, cp, I, L in [(64, 8, 2, 8, 32768), (1, 1, 1, 1, 1), (3, 2, 4, 8, 1000),
                             (64, 8, 2, 8, 1024), (2, 8, 8, 16, 5)]:
        ns, st = ctypes.c_int32(), ctypes.c_int32()
        assert lib.cp_decode_plan(B, Hkv, cp, I, 16, L, ctypes.byref(ns), ctypes.byref(st)) == 0
        group = I * cp
        share = (L // group) * I + min(L % group, I)
        assert st.value % 16 == 0 and ns.value * st.value >= share
        assert (ns.value - 1) * st.value < max(share, 1)


def test_prefill_mode_selector_follows_its_measured_table(lib):
    """The selector returns the mode measured faster on one GB300 at the nearest grid point:
    pass-Q only where it won by more than 3% (q_len ~ 256 with kv_len ~ 2 q_len; G = 1 with
    q_len ~ 4096 and kv_len up to ~8 q_len), pass-KV elsewhere, including full prefill."""
    sel = lib.cp_select_prefill_mode
    assert sel(8192, 8192, 16, 2, 128, 2) == 0          # full prefill, G = 8
    assert sel(2048, 32768, 16, 2, 128, 2) == 0         # the chunked workload: within 1%
    for G in (1, 2, 4, 8, 16):
        assert sel(256, 512, 2 * G, 2, 128, 2) == 1      # q_len 256, kv_len = 2 q_len
        assert sel(256, 4096, 2 * G, 2, 128, 2) == 0
        assert sel(1024, 2048, 2 * G, 2, 128, 2) == 0
    assert sel(4096, 4096 * 4, 2, 2, 128, 2) == 1       # G = 1, q_len 4096, ratio 4
    assert sel(4096, 4096 * 32, 2, 2, 128, 2) == 0
    assert sel(4096, 4096 * 4, 4, 2, 128, 2) == 0       # G = 2
    assert sel(300, 560, 8, 2, 128, 2) == 1             # nearest grid point (256, 2, G = 4)
    assert sel(10, 5, 8, 2, 128, 2) == 0                # kv shorter than q: no pass-Q answer
