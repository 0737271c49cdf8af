#!/usr/bin/env python3
"""Throughput of the CP partial-attention hot path on one GB300 (and N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic input:
  prefill workloads (full, long, tiny): cp_partition -> cp_partial_attn_prefill (pass-KV)
      -> cp_lse_merge;
  chunked: cp_partition of the new tokens -> cp_kv_interleave_layout -> pass-Q partial
      attention -> cp_lse_merge;
  decode: cp_kv_interleave_layout -> cp_partial_attn_decode -> cp_lse_merge.
Default workload: full prefill (1 x 8192 tokens, 16/2 heads, d=128, bf16, cp=2), metric
causal TFLOP/s (4*d*Hq per visible (q, k) pair).  A decode measurement (GB/s of kv read) is
added as "secondary".  Multi-GPU: every rank runs an independent replica (CP shards are logical,
on one GPU each) -- weak scaling, no collective on the data path.

--impl reference times the float64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the dominant kernels,
# each from one ncu capture summarised under profiles/.  A figure is reported only while the
# kernel's source file still has the SHA-1 the capture was taken on; otherwise traffic is null.
NCU_TRAFFIC = {
    # profiles/prefill_tc2_full_prefill.md: dram read 42.04 MB + write 62.57 MB
    "prefill": {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                "sha1": "f72141077f3eace2e0309ce3d75b4c80a82e1d37", "bytes": 104614400,
                "workload": "full"},
    # profiles/decode_mma_decode.md: a 16-sequence capture (1.1187 GB read + 5.36 MB written),
    # scaled to the 64-sequence workload by algorithmic bytes (4.3933e9 / 1.1181e9)
    "decode": {"file": "context_gqa_attention_gb300/csrc/decode.cu",
               "sha1": "9b0d529eacd73ab4391495a21d18a2e537d1c074", "bytes": 4416620000,
               "workload": "decode"},
}

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 * 1024 * 1024


# ------------------------------------------------------------------------------------- utils

def ncu_traffic(kind, workload):
    import hashlib
    rec = NCU_TRAFFIC.get(kind)
    if not rec or rec.get("workload") != workload:
        return None
    path = os.path.join(ROOT, rec["file"])
    with open(path, "rb") as f:
        if hashlib.sha1(f.read()).hexdigest() != rec["sha1"]:
            return None
    return rec["bytes"]


def source_sha1():
    """SHA-1 over the library's sources (kernels, host code, header): names the exact build a
    line was measured on (a copied tree need not carry git metadata)."""
    import glob
    import hashlib
    h = hashlib.sha1()
    files = sorted(glob.glob(os.path.join(ROOT, "context_gqa_attention_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "cpattn.h"))
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        def pick(*keys):
            for k in keys:
                if isinstance(d.get(k), (int, float)):
                    return float(d[k]), "measured"
            return None
        hbm = pick("hbm_gbs")
        tf = pick("bf16_tflops")
        tfs = pick("bf16_tflops_sustained")
        return {"hbm": hbm or (FALLBACK_HBM_GBS, "fallback"),
                "bf16": tf or (FALLBACK_BF16_TFLOPS, "fallback"),
                "bf16_sustained": tfs or tf or (FALLBACK_BF16_TFLOPS, "fallback")}
    return {"hbm": (FALLBACK_HBM_GBS, "fallback"), "bf16": (FALLBACK_BF16_TFLOPS, "fallback"),
            "bf16_sustained": (FALLBACK_BF16_TFLOPS, "fallback")}


class ClockSampler:
    """nvidia-smi samples (200 ms) kept with host timestamps; summarised over a window."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.time(), [x.strip() for x in line.split(",")]))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 <= t <= t1]
        note = "in window"
        if not rows and self.samples:
            mid = 0.5 * (t0 + t1)
            rows = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
            note = "nearest sample (timed region shorter than the 200 ms sampling period)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w": statistics.median(pw) if pw else None, "samples": len(rows),
                "note": note}


# ------------------------------------------------------------------------------------- runners

def causal_pairs_pass_kv(lens):
    return sum(T * (T + 1) // 2 for T in lens)


def run_with_side_maps(runner, maps, attention):
    """One step: the map kernels (`maps`) on a side stream, concurrent with the attention
    kernels (`attention`) on the current stream, which derive their chunk bounds / rank
    lengths themselves; the side stream is joined before the step ends."""
    main = torch.cuda.current_stream(runner.dev)
    if getattr(runner, "s_side", None) is None:
        runner.s_side = torch.cuda.Stream(runner.dev)
    side = runner.s_side
    side.wait_stream(main)
    with torch.cuda.stream(side):
        maps()
    try:
        attention()
    finally:
        main.wait_stream(side)


class PrefillRunner:
    """pass-KV prefill: partition -> partial attention -> merge."""

    def __init__(self, w, dev, cpa):
        self.w, self.dev, self.cpa = w, dev, cpa
        lens = [w.seq_len] * w.num_seqs
        x = wl.prefill_inputs(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype, w.seed)
        self.host = {k: v.pin_memory() for k, v in x.items()}
        self.lens = lens
        self.N = sum(lens)
        self.q = x["q"].to(dev)
        self.k = x["k"].to(dev)
        self.v = x["v"].to(dev)
        self.cu = x["cu_seqlens"].to(dev)
        self.sets = None  # end-to-end: two device buffer sets, filled on first use
        cp, Hq, d = w.cp, w.num_q_heads, w.head_dim
        self.part = torch.empty(cp, self.N, Hq, d, dtype=torch.float32, device=dev)
        self.plse = torch.empty(cp, self.N, Hq, dtype=torch.float32, device=dev)
        self.out = torch.empty(self.N, Hq, d, dtype=w.dtype, device=dev)
        self.olse = torch.empty(self.N, Hq, dtype=torch.float32, device=dev)
        self.perm = torch.empty(self.N, dtype=torch.int32, device=dev)
        self.inv = torch.empty(self.N, dtype=torch.int32, device=dev)
        self.so = torch.empty(cp + 1, dtype=torch.int32, device=dev)
        self.cb = torch.empty(len(lens), 2 * cp + 1, dtype=torch.int32, device=dev)
        self.flops = 4.0 * d * Hq * causal_pairs_pass_kv(lens)
        self.impl = cpa.CP_IMPL_AUTO
        self.fused = False
        self.out_host = torch.empty(self.out.shape, dtype=w.dtype).pin_memory()

    def step(self, ev=None):
        cpa, w = self.cpa, self.w
        run_with_side_maps(
            self, lambda: cpa.cp_partition(self.cu, w.cp, self.N, self.perm, self.inv, self.so,
                                           self.cb),
            lambda: self._attention(ev))

    def _attention(self, ev=None):
        cpa, w = self.cpa, self.w
        if self.fused:  # every kv shard walked inside one item: final output, no partials
            if ev is not None:
                ev[0].record()
            cpa.cp_attn_prefill_fused(self.q, self.cu, w.cp, self.k, self.v,
                                      max_seqlen_q=max(self.lens), out=self.out, out_lse=self.olse,
                                      impl=self.impl)
            if ev is not None:
                ev[1].record()
            return
        if ev is not None:
            ev[0].record()
        cpa.cp_partial_attn_prefill(self.q, self.cu, w.cp, k=self.k, v=self.v,
                                    max_seqlen_q=max(self.lens), out=self.part, lse=self.plse,
                                    impl=self.impl)
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(self.part, self.plse, out=self.out, out_lse=self.olse)

    @property
    def launches_per_step(self):
        return 2 if self.fused else 3

    def _use(self, st):
        self.q, self.k, self.v, self.cu, self.out, self.olse = (
            st["q"], st["k"], st["v"], st["cu_seqlens"], st["out"], st["olse"])

    def e2e_run(self, steps, stream):
        """Host buffers in, host result out, every step: pinned host -> device copies of the
        step's inputs on one copy stream, the step on `stream`, its output copied back on a
        second copy stream.  Two device buffer sets let step i+1's inputs arrive and step
        i-1's output leave while step i computes (event-ordered).  Returns seconds."""
        dev = self.dev
        if self.sets is None:
            base = {"q": self.q, "k": self.k, "v": self.v, "cu_seqlens": self.cu,
                    "out": self.out, "olse": self.olse}
            other = {k: torch.empty_like(t) for k, t in base.items()}
            self.sets = [base, other]
            self.outs_host = [self.out_host, torch.empty_like(self.out_host).pin_memory()]
            self.s_in = torch.cuda.Stream(dev)
            self.s_out = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_ready = [ev(), ev()]
        in_free = [None, None]   # compute finished reading set b
        out_ready = [ev(), ev()]
        out_free = [None, None]  # output of set b copied to the host
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        self.s_in.wait_stream(stream)
        self.s_out.wait_stream(stream)
        for i in range(steps):
            b = i % 2
            st = self.sets[b]
            with torch.cuda.stream(self.s_in):
                if in_free[b] is not None:
                    self.s_in.wait_event(in_free[b])
                for name in ("q", "k", "v", "cu_seqlens"):
                    st[name].copy_(self.host[name], non_blocking=True)
                in_ready[b].record(self.s_in)
            stream.wait_event(in_ready[b])
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            self._use(st)
            self.step()
            done = ev()
            done.record(stream)
            in_free[b] = done
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(done)
                self.outs_host[b].copy_(st["out"], non_blocking=True)
                out_ready[b].record(self.s_out)
            out_free[b] = out_ready[b]
            out_ready[b] = ev()
        stream.wait_stream(self.s_in)
        stream.wait_stream(self.s_out)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        self.e2e_last = self.outs_host[(steps - 1) % 2]
        self._use(self.sets[0])
        return t0.elapsed_time(t1) / 1e3

    def e2e_check(self):
        """The host copy of the last pipelined step equals a fresh device-only step."""
        self.step()
        torch.cuda.synchronize(self.dev)
        return bool(torch.equal(self.out.cpu(), self.e2e_last))

    def e2e_bytes(self):
        h2d = sum(t.numel() * t.element_size() for t in self.host.values())
        return h2d, self.out.numel() * self.out.element_size()

    def metric(self, seconds):
        return self.flops / seconds / 1e12

    def config(self):
        return prefill_config(self.w)


def prefill_config(w):
    return {"workload": f"{w.name} prefill pass-KV: {w.num_seqs}x{w.seq_len} tokens, "
                        f"{w.num_q_heads}/{w.num_kv_heads} heads, d={w.head_dim}, cp={w.cp}",
            "seq_len": w.seq_len, "global_batch": w.num_seqs, "cp": w.cp,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "mode": "pass_kv"}


class PassQRunner:
    """chunked prefill (pass-Q): partition of the new tokens -> round-robin layout of the kv
    -> pass-Q partial attention over the paged cache -> merge."""

    def __init__(self, w, dev, cpa):
        self.w, self.dev, self.cpa = w, dev, cpa
        x = wl.workload_inputs(w)
        self.q = x["q"].to(dev)
        self.kc = x["k_cache"].to(dev)
        self.vc = x["v_cache"].to(dev)
        self.tables = x["block_tables"].to(dev)
        self.seq_lens = x["seq_lens"].to(dev)
        self.cu_q = x["cu_seqlens_q"].to(dev)
        cu = [0]
        for L in x["seq_lens"].tolist():
            cu.append(cu[-1] + L)
        self.cu_kv = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.N = w.num_seqs * w.q_len
        cp, Hq, d = w.cp, w.num_q_heads, w.head_dim
        self.part = torch.empty(cp, self.N, Hq, d, dtype=torch.float32, device=dev)
        self.plse = torch.empty(cp, self.N, Hq, dtype=torch.float32, device=dev)
        self.out = torch.empty(self.N, Hq, d, dtype=w.dtype, device=dev)
        self.local_lens = torch.empty(cp, w.num_seqs, dtype=torch.int32, device=dev)
        self.perm = torch.empty(self.N, dtype=torch.int32, device=dev)
        self.inv = torch.empty(self.N, dtype=torch.int32, device=dev)
        self.so = torch.empty(cp + 1, dtype=torch.int32, device=dev)
        self.cb = torch.empty(w.num_seqs, 2 * cp + 1, dtype=torch.int32, device=dev)
        ctx = w.kv_len - w.q_len
        pairs = sum(ctx + i + 1 for i in range(w.q_len)) * w.num_seqs
        self.flops = 4.0 * d * Hq * pairs
        self.impl = cpa.CP_IMPL_AUTO
        self.fused = False
        self.olse = torch.empty(self.N, Hq, dtype=torch.float32, device=dev)

    def step(self, ev=None):
        cpa, w = self.cpa, self.w

        def maps():
            cpa.cp_partition(self.cu_q, w.cp, self.N, self.perm, self.inv, self.so, self.cb)
            cpa.cp_kv_interleave_layout(self.cu_kv, w.cp, w.interleave, 0, w.block_size,
                                        local_lens=self.local_lens, want_slots=False)

        run_with_side_maps(self, maps, lambda: self._attention(ev))

    @property
    def launches_per_step(self):
        return 3 if self.fused else 4

    def _attention(self, ev=None):
        cpa, w = self.cpa, self.w
        if self.fused:  # every rank's resident pages walked inside one item: final output
            if ev is not None:
                ev[0].record()
            cpa.cp_attn_prefill_fused(self.q, self.cu_q, w.cp, mode=cpa.CP_PASS_Q,
                                      k_cache=self.kc, v_cache=self.vc, block_tables=self.tables,
                                      seq_lens_kv=self.seq_lens, interleave=w.interleave,
                                      max_seqlen_q=w.q_len, out=self.out, out_lse=self.olse,
                                      impl=self.impl)
            if ev is not None:
                ev[1].record()
            return
        if ev is not None:
            ev[0].record()
        cpa.cp_partial_attn_prefill(self.q, self.cu_q, w.cp, mode=cpa.CP_PASS_Q, k_cache=self.kc,
                                    v_cache=self.vc, block_tables=self.tables,
                                    seq_lens_kv=self.seq_lens, interleave=w.interleave,
                                    max_seqlen_q=w.q_len, out=self.part, lse=self.plse,
                                    impl=self.impl)
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(self.part, self.plse, out=self.out, want_lse=False)

    def metric(self, seconds):
        return self.flops / seconds / 1e12

    def config(self):
        w = self.w
        return {"workload": f"chunked prefill pass-Q: {w.num_seqs} seqs x {w.q_len} new of "
                            f"{w.kv_len} kv, {w.num_q_heads}/{w.num_kv_heads} heads, d={w.head_dim}, "
                            f"paged bs={w.block_size}, cp={w.cp}, I={w.interleave}",
                "mode": "pass_q"}


class DecodeRunner:
    """decode: interleave layout -> per-rank split partials -> merge."""

    def __init__(self, w, dev, cpa, on_device_values=True):
        self.w, self.dev, self.cpa = w, dev, cpa
        lens = wl.decode_lengths(w.num_seqs, w.min_len, w.max_len, w.len_seed).tolist()
        self.lens = lens
        caps = [wl.block_capacity(L, w.cp, w.interleave, w.block_size) for L in lens]
        tables, pool = wl.shuffled_block_tables(caps, w.cp, torch.Generator().manual_seed(w.table_seed))
        Hq, Hkv, d, cp = w.num_q_heads, w.num_kv_heads, w.head_dim, w.cp
        g = torch.Generator(device=dev).manual_seed(w.seed)
        shape = (cp, pool, Hkv, w.block_size, d)
        # kv values drawn on the device (same N(0,1) recipe; the bench checks no parity)
        self.kc = torch.randn(shape, generator=g, device=dev, dtype=w.dtype)
        self.vc = torch.randn(shape, generator=g, device=dev, dtype=w.dtype)
        self.q = torch.randn(w.num_seqs, Hq, d, generator=g, device=dev, dtype=w.dtype)
        self.tables = tables.to(dev)
        self.seq_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.ns, self.st = cpa.cp_decode_plan(w.num_seqs, Hkv, cp, w.interleave, w.block_size, max(lens))
        P = cp * self.ns
        self.part = torch.empty(P, w.num_seqs, Hq, d, dtype=torch.float32, device=dev)
        self.plse = torch.empty(P, w.num_seqs, Hq, dtype=torch.float32, device=dev)
        self.out = torch.empty(w.num_seqs, Hq, d, dtype=w.dtype, device=dev)
        self.fused = False  # two launches measured faster than the fused one
        self.ws = torch.zeros(cpa.cp_decode_workspace_size(w.num_seqs, Hq, Hkv, d, cp, self.ns),
                              dtype=torch.uint8, device=dev)
        self.local_lens = torch.empty(cp, w.num_seqs, dtype=torch.int32, device=dev)
        el = torch.tensor([], dtype=w.dtype).element_size()
        pages = sum(-(-n // w.block_size) for L in lens
                    for n in [(L // (w.interleave * cp)) * w.interleave
                              + min(max(L % (w.interleave * cp) - r * w.interleave, 0), w.interleave)
                              for r in range(cp)])
        self.bytes = (sum(lens) * Hkv * d * 2 * el + 2 * w.num_seqs * Hq * d * el + pages * 4)
        self.kv_bytes = sum(lens) * Hkv * d * 2 * el
        self.pool = pool

    def resplit(self, split_tokens):
        w = self.w
        share = self.ns * self.st  # the planned split covers the largest rank share
        self.st = split_tokens
        self.ns = -(-share // split_tokens)
        P = w.cp * self.ns
        Hq, d = w.num_q_heads, w.head_dim
        self.part = torch.empty(P, w.num_seqs, Hq, d, dtype=torch.float32, device=self.dev)
        self.plse = torch.empty(P, w.num_seqs, Hq, dtype=torch.float32, device=self.dev)
        self.ws = torch.zeros(self.cpa.cp_decode_workspace_size(w.num_seqs, Hq, w.num_kv_heads, d,
                                                                w.cp, self.ns),
                              dtype=torch.uint8, device=self.dev)

    @property
    def launches_per_step(self):
        return 2 if self.fused else 3

    def step(self, ev=None):
        cpa, w = self.cpa, self.w
        run_with_side_maps(
            self, lambda: cpa.cp_kv_interleave_layout(self.cu, w.cp, w.interleave, 0, w.block_size,
                                                      local_lens=self.local_lens, want_slots=False),
            lambda: self._attention(ev))

    def _attention(self, ev=None):
        cpa, w = self.cpa, self.w
        if ev is not None:
            ev[0].record()
        if self.fused:  # partials + merge in one launch
            cpa.cp_decode_attention(self.q, self.kc, self.vc, self.tables, self.seq_lens, w.cp,
                                    w.interleave, num_splits=self.ns, split_tokens=self.st,
                                    workspace=self.ws, out=self.out, want_lse=False)
            if ev is not None:
                ev[1].record()
            return
        cpa.cp_partial_attn_decode(self.q, self.kc, self.vc, self.tables, self.seq_lens, w.cp,
                                   w.interleave, num_splits=self.ns, split_tokens=self.st,
                                   out=self.part, lse=self.plse)
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(self.part, self.plse, out=self.out, want_lse=False)

    def e2e_run(self, steps, stream):
        """Every step copies its per-step inputs from pinned host memory (new query tokens,
        sequence lengths, block tables, cumulative lengths; the paged kv cache stays resident,
        as it would in serving) and reads the merged output back.  Returns seconds."""
        if not hasattr(self, "host"):
            self.host = {n: t.cpu().pin_memory() for n, t in
                         (("q", self.q), ("seq_lens", self.seq_lens), ("tables", self.tables),
                          ("cu", self.cu))}
            self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            for n in ("q", "seq_lens", "tables", "cu"):
                getattr(self, n).copy_(self.host[n], non_blocking=True)
            self.step()
            self.out_host.copy_(self.out, non_blocking=True)
        t1.record(stream)
        torch.cuda.synchronize(self.dev)
        return t0.elapsed_time(t1) / 1e3

    def e2e_bytes(self):
        h2d = sum(t.numel() * t.element_size() for t in self.host.values())
        return h2d, self.out.numel() * self.out.element_size()

    def e2e_check(self):
        last = self.out_host.clone()
        self.step()
        torch.cuda.synchronize(self.dev)
        return bool(torch.equal(self.out.cpu(), last))

    def metric(self, seconds):
        return self.bytes / seconds / 1e9

    def config(self):
        w = self.w
        return {"workload": f"decode: {w.num_seqs} seqs, ctx U[{w.min_len},{w.max_len}] "
                            f"(sum {sum(self.lens)}), {w.num_q_heads}/{w.num_kv_heads} heads, "
                            f"d={w.head_dim}, paged bs={w.block_size}, cp={w.cp}, I={w.interleave}",
                "splits": self.ns, "split_tokens": self.st}


def time_steps(runner, steps, warmup, flush, dev, stream, dominant=True, stretch_s=0.0):
    """Per-step device time (CUDA events on the launching stream), L2 flushed between steps."""
    for _ in range(warmup):
        flush.zero_()
        runner.step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dom = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if dominant else [None] * steps
    extra = 0
    if stretch_s > 0:  # extra flush passes keep the GPU busy so clocks can be sampled
        t = time.time()
        for _ in range(20):
            flush.zero_()
        torch.cuda.synchronize(dev)
        per_flush = max((time.time() - t) / 20, 1e-5)
        extra = int(max(0, stretch_s / steps / per_flush - 1))
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(steps):
        for _ in range(1 + extra):
            flush.zero_()
        torch.cuda.nvtx.range_push(f"{type(runner).__name__} step {i}")  # profiler timelines
        starts[i].record(stream)
        runner.step(dom[i])
        ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    t1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dom_ms = [a.elapsed_time(b) for a, b in dom] if dominant else []
    return step_ms, dom_ms, (t0, t1)


# ------------------------------------------------------------------------------------- oracle

def oracle_sample(w, rows_per_step, seed):
    """Time the float64 oracle on a bounded, stratified sample of query rows of the workload."""
    from oracle import cp_oracle as orc
    lens = [w.seq_len] * w.num_seqs
    x = wl.prefill_inputs(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype, w.seed)
    bnd = orc.chunk_bounds(w.seq_len, w.cp).tolist()
    rows = wl.sample_rows(w.seq_len, bnd, rows_per_step, seed)
    t = time.time()
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], w.cp,
                                1 / math.sqrt(w.head_dim), rows=rows)
    Om, Lm = orc.lse_merge(O, L)
    dt = time.time() - t
    flops = 4.0 * w.head_dim * w.num_q_heads * sum(r + 1 for r in rows)
    return flops, dt, len(rows), (rows, Om, Lm)


def parity_line(runner, ref):
    """Max errors of the bench's own merged output (the last device-only step) against the
    oracle rows the CPU baseline computed (same seeded inputs)."""
    import numpy as np
    rows, Om, Lm = ref
    idx = torch.as_tensor(rows, dtype=torch.long, device=runner.out.device)
    out = runner.out.index_select(0, idx).double().cpu().numpy()
    lse = runner.olse.index_select(0, idx).double().cpu().numpy()
    fin = np.isfinite(Lm)
    return {"rows": len(rows), "max_abs_out": float(np.abs(out - Om).max()),
            "max_rel_lse": float((np.abs(lse[fin] - Lm[fin]) / np.abs(Lm[fin]).clip(1e-30)).max()),
            "tolerance": "out 1e-2 + bf16 rounding 2^-8 |O|; lse 1e-3 relative"}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------------------------- main

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, dev):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    if w.kind != "pass_kv":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle reference arm times "
                                                             "prefill workloads only"}))
        return 0
    rows = args.ref_rows
    for i in range(args.warmup):
        oracle_sample(w, max(rows // 8, 8), 9000 + i)
    tot_flops, tot_t, nrows = 0.0, 0.0, 0
    for i in range(args.steps):
        f, t, n, _ = oracle_sample(w, rows, 9100 + i)
        tot_flops += f
        tot_t += t
        nrows += n
    val = tot_flops / tot_t / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": "causal GQA prefill TFLOP/s (pass-KV partial attention + LSE merge)",
        "value": val, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(w),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} stratified query rows x all heads per step "
                                   f"({nrows} rows total), float64 NumPy oracle"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full", choices=["full", "long", "tiny", "chunked", "decode"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=256)
    # cpu baseline: every query row of the full workload (~8-10 s of float64 oracle work)
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--prefill-impl", default="auto", choices=["auto", "tcgen05", "simt"])
    ap.add_argument("--prefill-fused", action="store_true",
                    help="prefill as one launch (cp_attn_prefill_fused) instead of partials + merge")
    ap.add_argument("--decode-fused", action="store_true",
                    help="decode as one launch (cp_decode_attention) instead of partials + merge")
    ap.add_argument("--decode-split-tokens", type=int, default=0,
                    help="override the decode plan's rank-local tokens per split (multiple of 16)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's number of sequences (smaller profiling cases)")
    ap.add_argument("--cp", type=int, default=0, help="override the number of logical CP ranks")
    ap.add_argument("--interleave", type=int, default=0, help="override the interleave size")
    ap.add_argument("--seed", type=int, default=-1, help="override the value seed")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import context_gqa_attention_gb300 as cpa
    cpa.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    w = wl.WORKLOADS[args.workload]
    if args.batch > 0:
        w = dataclasses.replace(w, num_seqs=args.batch)
    if args.cp > 0:
        w = dataclasses.replace(w, cp=args.cp)
    if args.interleave > 0:
        w = dataclasses.replace(w, interleave=args.interleave)
    if args.seed >= 0:
        w = dataclasses.replace(w, seed=args.seed)
    runner = (DecodeRunner(w, dev, cpa) if w.kind == "decode" else
              PassQRunner(w, dev, cpa) if w.kind == "pass_q" else PrefillRunner(w, dev, cpa))
    if isinstance(runner, DecodeRunner):
        runner.fused = args.decode_fused
        if args.decode_split_tokens > 0:
            runner.resplit(args.decode_split_tokens)
    if isinstance(runner, (PrefillRunner, PassQRunner)):
        runner.fused = args.prefill_fused
    runner.impl = {"auto": cpa.CP_IMPL_AUTO, "tcgen05": cpa.CP_IMPL_TCGEN05,
                   "simt": cpa.CP_IMPL_SIMT}[args.prefill_impl]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize(dev)
    step_ms, dom_ms, (t0, t1) = time_steps(runner, args.steps, args.warmup, flush, dev, stream,
                                           stretch_s=1.0)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.summary(t0, t1)
    clocks.stop()

    total_s = max_over_ranks(sum(step_ms) / 1e3, ws, dev)
    value = runner.metric(total_s / args.steps) * ws
    dom_s = statistics.mean(dom_ms) / 1e3

    # end to end: host buffers, copies inside the timed region
    if isinstance(runner, PassQRunner):
        e2e = None
        peak, src = pk["bf16"]
        achieved = runner.flops / dom_s / 1e12
        roof = {"bound": "tensor", "kernel": "cp_attn_prefill_fused (pass-Q, paged, merged in-kernel)"
                if runner.fused else "cp_partial_attn_prefill (pass-Q, paged)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{src} bf16 dense (burst)", "traffic": None,
                "algorithmic": f"{runner.flops:.4e} causal FLOP per launch", "launch_ms": dom_s * 1e3}
        metric = ("causal GQA chunked-prefill TFLOP/s (pass-Q, ranks merged in-kernel)" if runner.fused
                  else "causal GQA chunked-prefill TFLOP/s (pass-Q partial attention + LSE merge)")
        unit = "TFLOP/s"
    elif isinstance(runner, PrefillRunner):
        runner.e2e_run(3, stream)
        e2e_s = max_over_ranks(runner.e2e_run(args.steps, stream), ws, dev)
        if not runner.e2e_check():
            raise RuntimeError("end-to-end output differs from the device-only step")
        h2d, d2h = runner.e2e_bytes()
        e2e = {"value": runner.metric(e2e_s / args.steps) * ws, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelining": "inputs of step i+1 and output of step i-1 copied on two copy "
                             "streams while step i computes (double-buffered device sets)",
               "checked": "last host output == device-only step (bitwise)"}
        peak, src = pk["bf16"]
        achieved = runner.flops / dom_s / 1e12
        roof = {"bound": "tensor", "kernel": "cp_attn_prefill_fused (pass-KV, merged in-kernel)"
                if runner.fused else "cp_partial_attn_prefill (pass-KV)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{src} bf16 dense (burst)",
                "traffic": ncu_traffic("prefill", w.name),
                "algorithmic": f"{runner.flops:.4e} causal FLOP per launch",
                "launch_ms": dom_s * 1e3}
        metric = ("causal GQA prefill TFLOP/s (pass-KV, shards merged in-kernel)" if runner.fused
                  else "causal GQA prefill TFLOP/s (pass-KV partial attention + LSE merge)")
        unit = "TFLOP/s"
    else:
        runner.e2e_run(3, stream)
        e2e_s = max_over_ranks(runner.e2e_run(args.steps, stream), ws, dev)
        if not runner.e2e_check():
            raise RuntimeError("end-to-end output differs from the device-only step")
        h2d, d2h = runner.e2e_bytes()
        e2e = {"value": runner.metric(e2e_s / args.steps) * ws, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "checked": "last host output == device-only step (bitwise)"}
        peak, src = pk["hbm"]
        achieved = runner.bytes / dom_s / 1e9
        roof = {"bound": "hbm", "kernel": "cp_partial_attn_decode", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{src} HBM copy", "traffic": ncu_traffic("decode", w.name),
                "launch_ms": dom_s * 1e3,
                "algorithmic": f"{runner.bytes:.4e} B per launch (KV once + q + out + tables)"}
        metric = "decode KV-read GB/s (partial attention + LSE merge)"
        roof["kernel"] = "cp_decode_attention (fused partials + merge)" if runner.fused else roof["kernel"]
        unit = "GB/s"

    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": dict(runner.config(), l2="flushed between timed steps (512 MB write)",
                           parallelism=f"replicas x{ws} (logical CP shards on each GPU)"),
            "roofline": roof, "clocks": clk,
            "gpu_launches": runner.launches_per_step * args.steps,
            "source_sha1": source_sha1()}
    if e2e is not None:
        line["e2e"] = e2e

    if not args.no_secondary and w.kind != "decode":
        sec = {}
        if (isinstance(runner, PrefillRunner) and not isinstance(runner, PassQRunner)
                and w.dtype == torch.bfloat16):  # the fused launch takes bf16
            # the same workload as one launch (cp_attn_prefill_fused): no partial round trip
            runner.fused = not runner.fused
            fs, fd, _ = time_steps(runner, max(10, args.steps // 2), 3, flush, dev, stream)
            f_s = statistics.mean(fd) / 1e3
            bf, bsrc = pk["bf16"]
            sec["prefill_fused" if runner.fused else "prefill_partials"] = {
                "value": runner.metric(statistics.mean(fs) / 1e3), "unit": "TFLOP/s",
                "roofline": {"bound": "tensor",
                             "kernel": "cp_attn_prefill_fused" if runner.fused else
                             "cp_partial_attn_prefill (pass-KV)",
                             "achieved": runner.flops / f_s / 1e12, "peak": bf, "unit": "TFLOP/s",
                             "frac": runner.flops / f_s / 1e12 / bf,
                             "peak_source": f"{bsrc} bf16 dense (burst)", "launch_ms": f_s * 1e3}}
            runner.fused = not runner.fused
        hbm, hsrc = pk["hbm"]
        for fused in (False, True):
            dr = DecodeRunner(wl.WORKLOADS["decode"], dev, cpa)
            dr.fused = fused
            ds, dd, _ = time_steps(dr, max(10, args.steps // 5), 3, flush, dev, stream)
            d_s = statistics.mean(dd) / 1e3
            sec["decode_fused" if fused else "decode"] = {
                "value": dr.metric(statistics.mean(ds) / 1e3), "unit": "GB/s",
                "config": dr.config(),
                "roofline": {"bound": "hbm",
                             "kernel": "cp_decode_attention (partials + merge, one launch)" if fused
                             else "cp_partial_attn_decode (+ cp_lse_merge)",
                             "achieved": dr.bytes / d_s / 1e9, "peak": hbm,
                             "unit": "GB/s", "frac": dr.bytes / d_s / 1e9 / hbm,
                             "peak_source": f"{hsrc} HBM copy", "launch_ms": d_s * 1e3}}
            del dr
        line["secondary"] = sec

    if rank == 0 and ws == 1 and not args.no_cpu_baseline and w.kind == "pass_kv":
        f, t, n, ref = oracle_sample(w, args.cpu_rows, 777)
        if isinstance(runner, PrefillRunner) and not runner.fused:
            line["parity"] = parity_line(runner, ref)
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
                                "cpu_count": os.cpu_count(), "seconds": t,
                                "rows_per_s": n * w.num_q_heads / t,
                                "kind": "oracle",
                                "sample": (f"all {n} query rows" if n >= w.seq_len * w.num_seqs
                                           else f"{n} stratified query rows")
                                          + f" x {w.num_q_heads} heads of the {w.name} workload, "
                                          f"float64 NumPy oracle, {t:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
