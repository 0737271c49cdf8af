"""Python binding of libcpattn (include/cpattn.h): causal GQA partial attention over logical
context-parallel shards, LSE merge and the CP layout maps, on one GB300 (sm_103a).

Argument marshalling only: every function below checks tensor placement, dtype and shape,
then calls the C entry point of the same name on the current torch CUDA stream.  All the
arithmetic runs in the library's CUDA kernels; there is no fallback.  A missing or unbuilt
library raises ``CPError``.

PyTorch provides device memory and streams.  Output tensors may be passed in (the library
never allocates); when omitted they are allocated here with ``torch.empty``.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
import threading

import torch

from . import _build

__all__ = [
    "CPError", "load", "lib_path", "CP_F32", "CP_BF16", "CP_PASS_KV", "CP_PASS_Q",
    "CP_IMPL_AUTO", "CP_IMPL_TCGEN05", "CP_IMPL_SIMT", "CP_IMPL_TCGEN05_SINGLE",
    "cp_partition", "cp_kv_interleave_layout",
    "cp_partial_attn_prefill", "cp_decode_plan", "cp_partial_attn_decode", "cp_lse_merge",
    "cp_decode_workspace_size", "cp_decode_attention", "cp_decode_attention_noalloc",
    "cp_kv_cache_write", "cp_select_prefill_mode", "cp_attn_prefill_fused",
    "cp_prefill_fused_workspace_size", "STATUS",
]

CP_F32, CP_BF16 = 0, 1
CP_PASS_KV, CP_PASS_Q = 0, 1
CP_IMPL_AUTO, CP_IMPL_TCGEN05, CP_IMPL_SIMT, CP_IMPL_TCGEN05_SINGLE = 0, 1, 2, 3
STATUS = {0: "CP_OK", 1: "CP_ERR_INVALID_ARG", 2: "CP_ERR_UNSUPPORTED", 3: "CP_ERR_CUDA",
          4: "CP_ERR_TIMEOUT", 5: "CP_ERR_DEVICE_BOUNDS"}

_c_int32_p = ctypes.c_void_p
_vp = ctypes.c_void_p


class CPError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status
        self.detail = detail


class PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32), ("dtype", ctypes.c_int32), ("impl", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("cp", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("cu_seqlens_q", _vp), ("seq_lens_kv", _vp), ("q", _vp), ("k", _vp), ("v", _vp),
        ("k_cache", _vp), ("v_cache", _vp), ("pool_pages", ctypes.c_int64),
        ("block_tables", _vp), ("max_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("interleave", ctypes.c_int32), ("q_shard", ctypes.c_int32), ("kv_shard", ctypes.c_int32),
        ("total_q", ctypes.c_int32), ("debug", ctypes.c_int32), ("out", _vp), ("lse", _vp),
        ("err", _vp), ("cu_seqlens_kv", _vp), ("total_kv", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("cp", ctypes.c_int32),
        ("interleave", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("num_splits", ctypes.c_int32), ("split_tokens", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("max_blocks", ctypes.c_int32),
        ("pool_pages", ctypes.c_int64), ("q", _vp), ("k_cache", _vp), ("v_cache", _vp),
        ("block_tables", _vp), ("seq_lens", _vp), ("out", _vp), ("lse", _vp), ("err", _vp),
    ]


_LIB = None

# (name, restype, argtypes)
_SIGS = [
    ("cp_status_string", ctypes.c_char_p, [ctypes.c_int32]),
    ("cp_last_error", ctypes.c_int32, [ctypes.c_char_p, ctypes.c_size_t]),
    ("cp_last_error_detail", ctypes.c_int32, [ctypes.c_char_p, ctypes.c_size_t]),
    ("cp_abi_version", ctypes.c_int32, []),
    ("cp_prefill_args_size", ctypes.c_size_t, []),
    ("cp_decode_args_size", ctypes.c_size_t, []),
    ("cp_partition", ctypes.c_int32, [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                      _vp, _vp, _vp, _vp]),
    ("cp_kv_interleave_layout", ctypes.c_int32, [_vp, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp,
                                                 _vp]),
    ("cp_kv_cache_write", ctypes.c_int32, [_vp, _vp, _vp, _vp] + [ctypes.c_int32] * 8 +
     [_vp, ctypes.c_int32, ctypes.c_int64, _vp, _vp, _vp, _vp]),
    ("cp_prefill_fused_workspace_size", ctypes.c_int32, [ctypes.POINTER(PrefillArgs),
                                                         ctypes.POINTER(ctypes.c_size_t)]),
    ("cp_attn_prefill_fused", ctypes.c_int32, [ctypes.POINTER(PrefillArgs), _vp, ctypes.c_size_t,
                                               _vp, _vp, _vp]),
    ("cp_select_prefill_mode", ctypes.c_int32, [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int32] * 4),
    ("cp_partial_attn_prefill", ctypes.c_int32, [ctypes.POINTER(PrefillArgs), _vp]),
    ("cp_decode_plan", ctypes.c_int32, [ctypes.c_int32] * 6 + [ctypes.POINTER(ctypes.c_int32)] * 2),
    ("cp_partial_attn_decode", ctypes.c_int32, [ctypes.POINTER(DecodeArgs), _vp]),
    ("cp_lse_merge", ctypes.c_int32, [_vp, _vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp]),
    ("cp_decode_workspace_size", ctypes.c_int32, [ctypes.c_int32] * 6 + [ctypes.POINTER(ctypes.c_size_t)]),
    ("cp_decode_attention", ctypes.c_int32, [ctypes.POINTER(DecodeArgs), _vp, ctypes.c_size_t, _vp,
                                             _vp, _vp]),
    ("cp_decode_attention_noalloc", ctypes.c_int32, [ctypes.POINTER(DecodeArgs), _vp, _vp, _vp]),
]

EXPORTED = [s[0] for s in _SIGS]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libcpattn.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise CPError(3, f"{path} is missing: build the CUDA library first "
                             "(python -c 'import __graft_entry__ as g; g.build()')")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, res, args in _SIGS:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.cp_prefill_args_size() != ctypes.sizeof(PrefillArgs):
        raise CPError(1, "cp_prefill_args layout mismatch between binding and library")
    if lib.cp_decode_args_size() != ctypes.sizeof(DecodeArgs):
        raise CPError(1, "cp_decode_args layout mismatch between binding and library")
    _LIB = lib
    return lib


def _check(st):
    if st != 0:
        buf = ctypes.create_string_buffer(512)
        _LIB.cp_last_error(buf, 512)
        raise CPError(st, buf.value.decode(errors="replace"))


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_CALL = threading.local()


def _on_first_tensors_device(fn):
    """Runs an entry point with its first tensor argument's device current (so the launch, the
    stream and any tensor allocated here belong to that device) and makes every other tensor
    argument check that it lives on the same device."""
    @functools.wraps(fn)
    def wrapper(first, *args, **kwargs):
        if not isinstance(first, torch.Tensor) or not first.is_cuda:
            raise CPError(1, f"{fn.__name__}: the first argument must be a CUDA tensor")
        prev = getattr(_CALL, "device", None)
        _CALL.device = first.device
        try:
            with torch.cuda.device(first.device):
                return fn(first, *args, **kwargs)
        finally:
            _CALL.device = prev
    return wrapper


def _dev(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise CPError(1, f"{name} must be a CUDA tensor")
    want = getattr(_CALL, "device", None)
    if want is not None and t.device != want:
        raise CPError(1, f"{name} is on {t.device} but the call runs on {want}: every tensor "
                         "of one call must be on the same device")
    if not t.is_contiguous():
        raise CPError(1, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise CPError(1, f"{name} must be {dtype} (got {t.dtype})")


def _kv_source(a, k, v, cu_seqlens_kv, dtype):
    """PASS_KV operands: k, v [Nkv, Hkv, d] and, for a cached context, cu_seqlens_kv [B + 1]."""
    _dev(k, "k", dtype)
    _dev(v, "v", dtype)
    if k is None or v is None or k.shape != v.shape:
        raise CPError(1, "PASS_KV needs k and v of the same shape [Nkv, Hkv, d]")
    a.num_kv_heads = k.shape[1]
    a.k, a.v = _ptr(k), _ptr(v)
    if cu_seqlens_kv is not None:
        _dev(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
        a.cu_seqlens_kv, a.total_kv = _ptr(cu_seqlens_kv), k.shape[0]


def _cp_dtype(t):
    if t.dtype == torch.bfloat16:
        return CP_BF16
    if t.dtype == torch.float32:
        return CP_F32
    raise CPError(2, f"unsupported dtype {t.dtype}")


# ------------------------------------------------------------------------------- entry points

@_on_first_tensors_device
def cp_partition(cu_seqlens, cp, total_tokens, perm=None, inv_perm=None, shard_offsets=None,
                 chunk_bounds=None, stream=None):
    """Load-balanced CP partition (see cpattn.h).  Returns (perm, inv_perm, shard_offsets,
    chunk_bounds) as int32 device tensors."""
    load()
    B = cu_seqlens.numel() - 1
    dev = cu_seqlens.device
    perm = torch.empty(total_tokens, dtype=torch.int32, device=dev) if perm is None else perm
    inv_perm = torch.empty(total_tokens, dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    shard_offsets = torch.empty(cp + 1, dtype=torch.int32, device=dev) if shard_offsets is None else shard_offsets
    chunk_bounds = torch.empty(B, 2 * cp + 1, dtype=torch.int32, device=dev) if chunk_bounds is None else chunk_bounds
    for n, t in (("cu_seqlens", cu_seqlens), ("perm", perm), ("inv_perm", inv_perm),
                 ("shard_offsets", shard_offsets), ("chunk_bounds", chunk_bounds)):
        _dev(t, n, torch.int32)
    _check(_LIB.cp_partition(_ptr(cu_seqlens), B, total_tokens, cp, _ptr(perm), _ptr(inv_perm),
                             _ptr(shard_offsets), _ptr(chunk_bounds), _stream(stream)))
    return perm, inv_perm, shard_offsets, chunk_bounds


@_on_first_tensors_device
def cp_kv_interleave_layout(cu_seq_lens, cp, interleave, total_tokens, block_size=16,
                            block_tables=None, local_lens=None, rank_of_token=None,
                            local_of_token=None, slot_of_token=None, want_slots=True, err=None,
                            stream=None):
    """Round-robin kv placement (see cpattn.h).  Returns (local_lens [cp, B], rank_of_token,
    local_of_token, slot_of_token-or-None)."""
    load()
    B = cu_seq_lens.numel() - 1
    dev = cu_seq_lens.device
    if local_lens is None:
        local_lens = torch.empty(cp, B, dtype=torch.int32, device=dev)
    if rank_of_token is None:
        rank_of_token = torch.empty(total_tokens, dtype=torch.int32, device=dev)
    if local_of_token is None:
        local_of_token = torch.empty(total_tokens, dtype=torch.int32, device=dev)
    if slot_of_token is None and want_slots and block_tables is not None:
        slot_of_token = torch.empty(total_tokens, dtype=torch.int64, device=dev)
    max_blocks = block_tables.shape[-1] if block_tables is not None else 0
    _dev(cu_seq_lens, "cu_seq_lens", torch.int32)
    _dev(block_tables, "block_tables", torch.int32)
    _check(_LIB.cp_kv_interleave_layout(
        _ptr(cu_seq_lens), B, total_tokens, cp, interleave, block_size, _ptr(block_tables),
        max_blocks, _ptr(local_lens), _ptr(rank_of_token), _ptr(local_of_token),
        _ptr(slot_of_token), _ptr(err), _stream(stream)))
    return local_lens, rank_of_token, local_of_token, slot_of_token


@_on_first_tensors_device
def cp_kv_cache_write(k_new, v_new, cu_new, start_pos, k_cache, v_cache, block_tables, cp,
                      interleave, err=None, stream=None):
    """Store new K/V rows [N, Hkv, d] into the per-rank pools [cp, pool, Hkv, bs, d] at their
    round-robin slots (see cpattn.h)."""
    load()
    N, Hkv, d = k_new.shape
    B = cu_new.numel() - 1
    for n, t, dt in (("k_new", k_new, None), ("v_new", v_new, k_new.dtype),
                     ("cu_new", cu_new, torch.int32), ("start_pos", start_pos, torch.int32),
                     ("k_cache", k_cache, k_new.dtype), ("v_cache", v_cache, k_new.dtype),
                     ("block_tables", block_tables, torch.int32)):
        _dev(t, n, dt)
    _check(_LIB.cp_kv_cache_write(_ptr(k_new), _ptr(v_new), _ptr(cu_new), _ptr(start_pos), B, N,
                                  Hkv, d, _cp_dtype(k_new), cp, interleave, k_cache.shape[3],
                                  _ptr(block_tables), block_tables.shape[-1], k_cache.shape[1],
                                  _ptr(k_cache), _ptr(v_cache), _ptr(err), _stream(stream)))


def cp_select_prefill_mode(q_len, kv_len, num_q_heads, num_kv_heads, head_dim, elem_bytes=2):
    """CP_PASS_KV or CP_PASS_Q: the mode measured faster on one GB300 for the nearest shape of a
    (q_len, kv_len, q heads per kv head) grid (see cpattn.h)."""
    load()
    return _LIB.cp_select_prefill_mode(q_len, kv_len, num_q_heads, num_kv_heads, head_dim,
                                       elem_bytes)


@_on_first_tensors_device
def cp_partial_attn_prefill(q, cu_seqlens_q, cp, *, mode=CP_PASS_KV, k=None, v=None,
                            cu_seqlens_kv=None, k_cache=None, v_cache=None, block_tables=None,
                            seq_lens_kv=None, interleave=8, max_seqlen_q=None, softmax_scale=0.0,
                            impl=CP_IMPL_AUTO, q_shard=-1, kv_shard=-1, out=None, lse=None,
                            err=None, debug=0, stream=None):
    """Partial attention of every (Q shard, KV shard) pair (see cpattn.h).

    q: [Nq, Hq, d].  PASS_KV: k, v [Nkv, Hkv, d]; with cu_seqlens_kv (int32 [B + 1]) each
    sequence's queries are the last of its kv tokens (a cached context before them), else
    Nkv = Nq and q, k, v share cu_seqlens_q.  PASS_Q: k_cache/v_cache [cp, pool, Hkv, 16, d],
    block_tables int32 [cp, B, max_blocks], seq_lens_kv int32 [B].
    Returns (out [cp, Nq, Hq, d] f32, lse [cp, Nq, Hq] f32).
    """
    load()
    Nq, Hq, d = q.shape
    B = cu_seqlens_q.numel() - 1
    dev = q.device
    if out is None:
        out = torch.empty(cp, Nq, Hq, d, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(cp, Nq, Hq, dtype=torch.float32, device=dev)
    a = PrefillArgs()
    a.mode, a.dtype, a.impl = mode, _cp_dtype(q), impl
    a.num_seqs, a.num_q_heads, a.head_dim, a.cp = B, Hq, d, cp
    a.softmax_scale = softmax_scale
    a.total_q = Nq
    a.q_shard, a.kv_shard = q_shard, kv_shard
    a.debug = debug
    _dev(q, "q")
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(out, "out", torch.float32)
    _dev(lse, "lse", torch.float32)
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    a.max_seqlen_q = max_seqlen_q
    a.cu_seqlens_q, a.q, a.out, a.lse, a.err = _ptr(cu_seqlens_q), _ptr(q), _ptr(out), _ptr(lse), _ptr(err)
    if mode == CP_PASS_KV:
        _kv_source(a, k, v, cu_seqlens_kv, q.dtype)
    else:
        _dev(k_cache, "k_cache", q.dtype)
        _dev(v_cache, "v_cache", q.dtype)
        _dev(block_tables, "block_tables", torch.int32)
        _dev(seq_lens_kv, "seq_lens_kv", torch.int32)
        a.num_kv_heads = k_cache.shape[2]
        a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
        a.pool_pages = k_cache.shape[1]
        a.block_tables, a.max_blocks = _ptr(block_tables), block_tables.shape[-1]
        a.block_size, a.interleave = k_cache.shape[3], interleave
        a.seq_lens_kv = _ptr(seq_lens_kv)
    _check(_LIB.cp_partial_attn_prefill(ctypes.byref(a), _stream(stream)))
    return out, lse


@_on_first_tensors_device
def cp_attn_prefill_fused(q, cu_seqlens_q, cp, k=None, v=None, *, mode=CP_PASS_KV,
                          cu_seqlens_kv=None, k_cache=None, v_cache=None, block_tables=None,
                          seq_lens_kv=None, interleave=8, max_seqlen_q=None, softmax_scale=0.0,
                          impl=CP_IMPL_AUTO, workspace=None, out=None, out_lse=None,
                          stream=None):
    """Prefill with the merge folded in (see cpattn.h): exact causal attention out [Nq, Hq, d]
    bf16 and lse [Nq, Hq] f32 without partials.  PASS_KV: k, v [Nkv, Hkv, d] (cu_seqlens_kv as
    in cp_partial_attn_prefill).  PASS_Q: the paged round-robin cache as in
    cp_partial_attn_prefill (every rank's resident tokens in one pass); `workspace` (uint8
    CUDA tensor of cp_prefill_fused_workspace_size() bytes) lets it split the tail wave's
    items by rank range; None allocates it, an empty tensor runs every item whole."""
    load()
    Nq, Hq, d = q.shape
    B = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty(Nq, Hq, d, dtype=torch.bfloat16, device=q.device)
    if out_lse is None:
        out_lse = torch.empty(Nq, Hq, dtype=torch.float32, device=q.device)
    for n, t, dt in (("q", q, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                     ("out", out, torch.bfloat16), ("out_lse", out_lse, torch.float32)):
        _dev(t, n, dt)
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    a = PrefillArgs()
    a.mode, a.dtype, a.impl = mode, CP_BF16, impl
    a.num_seqs, a.num_q_heads, a.head_dim, a.cp = B, Hq, d, cp
    a.softmax_scale, a.total_q, a.max_seqlen_q = softmax_scale, Nq, max_seqlen_q
    a.q_shard = a.kv_shard = -1
    a.cu_seqlens_q, a.q = _ptr(cu_seqlens_q), _ptr(q)
    if mode == CP_PASS_KV:
        _kv_source(a, k, v, cu_seqlens_kv, torch.bfloat16)
    else:
        for n, t, dt in (("k_cache", k_cache, torch.bfloat16), ("v_cache", v_cache, torch.bfloat16),
                         ("block_tables", block_tables, torch.int32),
                         ("seq_lens_kv", seq_lens_kv, torch.int32)):
            _dev(t, n, dt)
        a.num_kv_heads = k_cache.shape[2]
        a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
        a.pool_pages = k_cache.shape[1]
        a.block_tables, a.max_blocks = _ptr(block_tables), block_tables.shape[-1]
        a.block_size, a.interleave = k_cache.shape[3], interleave
        a.seq_lens_kv = _ptr(seq_lens_kv)
    if workspace is None:
        need = ctypes.c_size_t()
        _check(_LIB.cp_prefill_fused_workspace_size(ctypes.byref(a), ctypes.byref(need)))
        workspace = torch.empty(need.value, dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace")
    ws, ws_bytes = (_ptr(workspace), workspace.numel()) if workspace.numel() else (None, 0)
    _check(_LIB.cp_attn_prefill_fused(ctypes.byref(a), ws, ws_bytes, _ptr(out), _ptr(out_lse),
                                      _stream(stream)))
    return out, out_lse


def cp_prefill_fused_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, cp,
                                    max_seqlen_q, *, mode=CP_PASS_Q, impl=CP_IMPL_AUTO):
    """Bytes of workspace cp_attn_prefill_fused splits its tail wave with on the current device
    (0: no split for these shapes)."""
    load()
    a = PrefillArgs()
    a.mode, a.dtype, a.impl = mode, CP_BF16, impl
    a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.cp = (
        num_seqs, num_q_heads, num_kv_heads, head_dim, cp)
    a.max_seqlen_q, a.q_shard, a.kv_shard = max_seqlen_q, -1, -1
    need = ctypes.c_size_t()
    _check(_LIB.cp_prefill_fused_workspace_size(ctypes.byref(a), ctypes.byref(need)))
    return need.value


def cp_decode_plan(num_seqs, num_kv_heads, cp, interleave, block_size, max_seq_len):
    """(num_splits, split_tokens) for cp_partial_attn_decode."""
    load()
    ns, st = ctypes.c_int32(), ctypes.c_int32()
    _check(_LIB.cp_decode_plan(num_seqs, num_kv_heads, cp, interleave, block_size, max_seq_len,
                               ctypes.byref(ns), ctypes.byref(st)))
    return ns.value, st.value


@_on_first_tensors_device
def cp_partial_attn_decode(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave, *,
                           max_seq_len=None, num_splits=None, split_tokens=None, softmax_scale=0.0,
                           out=None, lse=None, err=None, stream=None):
    """Per-(rank, split) decode partials (see cpattn.h).  Returns (out [P, B, Hq, d], lse [P, B, Hq])
    with P = cp * num_splits."""
    load()
    B, Hq, d = q.shape
    Hkv, bs = k_cache.shape[2], k_cache.shape[3]
    if num_splits is None or split_tokens is None:
        if max_seq_len is None:
            max_seq_len = int(seq_lens.max().item())
        num_splits, split_tokens = cp_decode_plan(B, Hkv, cp, interleave, bs, max_seq_len)
    P = cp * num_splits
    if out is None:
        out = torch.empty(P, B, Hq, d, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(P, B, Hq, dtype=torch.float32, device=q.device)
    for n, t, dt in (("q", q, None), ("k_cache", k_cache, q.dtype), ("v_cache", v_cache, q.dtype),
                     ("block_tables", block_tables, torch.int32), ("seq_lens", seq_lens, torch.int32),
                     ("out", out, torch.float32), ("lse", lse, torch.float32)):
        _dev(t, n, dt)
    a = DecodeArgs()
    a.dtype, a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim = _cp_dtype(q), B, Hq, Hkv, d
    a.cp, a.interleave, a.block_size = cp, interleave, bs
    a.num_splits, a.split_tokens, a.softmax_scale = num_splits, split_tokens, softmax_scale
    a.max_blocks, a.pool_pages = block_tables.shape[-1], k_cache.shape[1]
    a.q, a.k_cache, a.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
    a.block_tables, a.seq_lens, a.out, a.lse, a.err = (_ptr(block_tables), _ptr(seq_lens), _ptr(out),
                                                       _ptr(lse), _ptr(err))
    _check(_LIB.cp_partial_attn_decode(ctypes.byref(a), _stream(stream)))
    return out, lse


def _decode_args(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave, num_splits,
                 split_tokens, softmax_scale, out, lse, err):
    B, Hq, d = q.shape
    for n, t, dt in (("q", q, None), ("k_cache", k_cache, q.dtype), ("v_cache", v_cache, q.dtype),
                     ("block_tables", block_tables, torch.int32), ("seq_lens", seq_lens, torch.int32)):
        _dev(t, n, dt)
    a = DecodeArgs()
    a.dtype, a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim = _cp_dtype(q), B, Hq, k_cache.shape[2], d
    a.cp, a.interleave, a.block_size = cp, interleave, k_cache.shape[3]
    a.num_splits, a.split_tokens, a.softmax_scale = num_splits, split_tokens, softmax_scale
    a.max_blocks, a.pool_pages = block_tables.shape[-1], k_cache.shape[1]
    a.q, a.k_cache, a.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
    a.block_tables, a.seq_lens, a.out, a.lse, a.err = (_ptr(block_tables), _ptr(seq_lens), _ptr(out),
                                                       _ptr(lse), _ptr(err))
    return a


def cp_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, cp, num_splits):
    """Bytes of scratch cp_decode_attention needs."""
    load()
    n = ctypes.c_size_t()
    _check(_LIB.cp_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, cp,
                                         num_splits, ctypes.byref(n)))
    return n.value


@_on_first_tensors_device
def cp_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave, *,
                        max_seq_len=None, num_splits=None, split_tokens=None, softmax_scale=0.0,
                        workspace=None, out=None, out_lse=None, want_lse=True, err=None,
                        stream=None):
    """Decode partials + merge in one launch (see cpattn.h).  `workspace` is a zero-filled
    uint8 CUDA tensor of at least cp_decode_workspace_size() bytes; it is left reusable.
    Returns (out [B, Hq, d] dtype of q, lse [B, Hq] f32 or None)."""
    load()
    B, Hq, d = q.shape
    Hkv, bs = k_cache.shape[2], k_cache.shape[3]
    if num_splits is None or split_tokens is None:
        if max_seq_len is None:
            max_seq_len = int(seq_lens.max().item())
        num_splits, split_tokens = cp_decode_plan(B, Hkv, cp, interleave, bs, max_seq_len)
    need = cp_decode_workspace_size(B, Hq, Hkv, d, cp, num_splits)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(B, Hq, d, dtype=q.dtype, device=q.device)
    if out_lse is None and want_lse:
        out_lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _dev(workspace, "workspace")
    _dev(out, "out", q.dtype)
    _dev(out_lse, "out_lse", torch.float32)
    a = _decode_args(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave, num_splits,
                     split_tokens, softmax_scale, None, None, err)
    _check(_LIB.cp_decode_attention(ctypes.byref(a), _ptr(workspace), workspace.numel(), _ptr(out),
                                    _ptr(out_lse), _stream(stream)))
    return out, out_lse


NOALLOC_SCRATCH_BYTES = 48 * 1024 * 1024


@_on_first_tensors_device
def cp_decode_attention_noalloc(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave,
                                out, *, num_splits, split_tokens, softmax_scale=0.0, out_lse=None,
                                err=None, stream=None):
    """cp_decode_attention for callers that cannot allocate device memory at call time.

    Scratch comes from a 48 MiB array built into the library (one per GPU, kept until the
    process exits), so neither this function nor the library allocates: the caller passes
    `out` ([B, Hq, d], dtype of q) and optionally `out_lse` ([B, Hq] f32), and the split plan
    explicitly (cp_decode_plan gives one).  Sizes that need more scratch than the array holds
    raise CPError (CP_ERR_INVALID_ARG).  Calls share the array, so calls that overlap on the GPU
    race; the first call on a device resolves the array's address and should come before any
    stream capture.
    """
    load()
    _dev(out, "out", q.dtype)
    _dev(out_lse, "out_lse", torch.float32)
    a = _decode_args(q, k_cache, v_cache, block_tables, seq_lens, cp, interleave, num_splits,
                     split_tokens, softmax_scale, None, None, err)
    _check(_LIB.cp_decode_attention_noalloc(ctypes.byref(a), _ptr(out), _ptr(out_lse),
                                            _stream(stream)))
    return out, out_lse


@_on_first_tensors_device
def cp_lse_merge(partial_out, partial_lse, out=None, out_dtype=torch.bfloat16, out_lse=None,
                 want_lse=True, stream=None):
    """Merge partials [P, rows, H, d] / [P, rows, H] into out [rows, H, d] (+ lse [rows, H])."""
    load()
    P, rows, H, d = partial_out.shape
    if out is None:
        out = torch.empty(rows, H, d, dtype=out_dtype, device=partial_out.device)
    if out_lse is None and want_lse:
        out_lse = torch.empty(rows, H, dtype=torch.float32, device=partial_out.device)
    _dev(partial_out, "partial_out", torch.float32)
    _dev(partial_lse, "partial_lse", torch.float32)
    _dev(out, "out")
    _dev(out_lse, "out_lse", torch.float32)
    _check(_LIB.cp_lse_merge(_ptr(partial_out), _ptr(partial_lse), P, rows, H, d, _ptr(out),
                             _cp_dtype(out), _ptr(out_lse), _stream(stream)))
    return out, out_lse


def default_scale(head_dim):
    return 1.0 / math.sqrt(head_dim)
