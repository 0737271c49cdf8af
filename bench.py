#!/usr/bin/env python3
"""Throughput of the CP partial-attention hot path on one GB300 (and N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic input:
  prefill workloads (long, full, tiny): cp_partition -> cp_partial_attn_prefill (pass-KV)
      -> cp_lse_merge;
  chunked: cp_partition of the new tokens -> cp_kv_interleave_layout -> pass-Q partial
      attention -> cp_lse_merge;
  decode: cp_kv_interleave_layout -> cp_partial_attn_decode -> cp_lse_merge.
Default workload: long prefill (2 x 32768 tokens, 16/2 heads, d=128, bf16, cp=4), metric causal
TFLOP/s (4*d*Hq per visible (q, k) pair).  The other workloads and forms are measured as
"secondary" entries, each with the roofline of its dominant kernel: full prefill, the fused
prefill launches, chunked pass-Q (partials and fused, end to end, parity), decode (two launches
and fused, end to end, parity) and the LSE merge alone.  Multi-GPU: every rank runs an
independent replica (CP shards are logical, on one GPU each) -- weak scaling, no collective on
the data path.

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

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a dominant kernel,
# each from one ncu capture (one pass, a warm launch: "-k regex:<kernel> -s 2 -c 1" on the bench
# command of that form, 3 warm-up steps) at the recorded source SHA-1.  A figure is reported only
# while that source file still has this SHA-1; otherwise traffic is null.
NCU_TRAFFIC = {
    # prefill_tc2_kernel<128,0,0,0>, pass-KV partials: dram read 42.03 MB + write 59.00 MB
    ("prefill", "full"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                         "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 101029632},
    # the same kernel, fused pass-KV: read 42.03 MB + write 1.17 MB (the bf16 output is still in L2)
    ("prefill_fused", "full"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                               "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 43200512},
    # long prefill partials: read 373.7 MB + write 1708.7 MB
    ("prefill", "long"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                         "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 2082401024},
    # long prefill fused: read 344.8 MB + write 234.3 MB
    ("prefill_fused", "long"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                               "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 579085312},
    # prefill_tc2_kernel<128,1,0,0>, pass-Q partials: read 172.1 MB + write 222.7 MB
    ("pass_q", "chunked"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                           "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 394838528},
    # prefill_tc2_kernel<128,1,0,1>, fused pass-Q (split tail): read 226.4 MB + write 24.8 MB
    ("pass_q_fused", "chunked"): {"file": "context_gqa_attention_gb300/csrc/prefill_tc.cu",
                                 "sha1": "e7cab9b56d6dd9a314e745bf2f0e2bc48b0516d5", "bytes": 251136512},
    # decode_mma_kernel<128,4,0>, 64-sequence decode: read 4.401 GB + write 23.6 MB
    ("decode", "decode"): {"file": "context_gqa_attention_gb300/csrc/decode.cu",
                          "sha1": "04b21175c45ac2e18e4f0cfc55d0f73c550df2ff", "bytes": 4425008128},
    # decode_mma_kernel<128,4,1> (fused merge): read 4.402 GB + write 16.1 MB
    ("decode_fused", "decode"): {"file": "context_gqa_attention_gb300/csrc/decode.cu",
                                "sha1": "04b21175c45ac2e18e4f0cfc55d0f73c550df2ff", "bytes": 4418197248},
}

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 * 1024 * 1024


# ------------------------------------------------------------------------------------- utils

def ncu_traffic(kind, workload):
    import hashlib
    rec = NCU_TRAFFIC.get((kind, workload))
    if not rec:
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


class Runner:
    """A step over device buffers `self.buf` (name -> tensor).  End to end, the names in
    `e2e_in` are copied from pinned host memory (`self.host`) every step and the names in
    `e2e_out` are read back, through two device buffer sets so that step i+1's inputs arrive
    and step i-1's outputs leave while step i computes (event-ordered copy streams)."""

    e2e_in = ()
    e2e_out = ("out",)
    e2e_note = ""

    def __init__(self, dev, cpa):
        self.dev, self.cpa = dev, cpa
        self.buf = {}
        self.host = {}
        self._sets = None
        self.e2e_mode = False  # a step of the end-to-end loop (e.g. also writes new kv)

    def e2e_prepare(self):
        """Pinned host copies of the step inputs (called once, outside any timed region)."""
        for n in self.e2e_in:
            if n not in self.host:
                self.host[n] = self.buf[n].cpu().pin_memory()

    def e2e_run(self, steps, stream):
        dev = self.dev
        self.e2e_prepare()
        if self._sets is None:
            names = list(self.e2e_in) + list(self.e2e_out)
            base = {n: self.buf[n] for n in names}
            other = {n: torch.empty_like(t) for n, t in base.items()}
            self._sets = [base, other]
            self._outs_host = [{n: torch.empty(self.buf[n].shape, dtype=self.buf[n].dtype).pin_memory()
                                for n in self.e2e_out} for _ in range(2)]
            self._s_in = torch.cuda.Stream(dev)
            self._s_out = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_ready = [ev(), ev()]
        in_free = [None, None]
        out_ready = [ev(), ev()]
        out_free = [None, None]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.e2e_mode = True
        t0.record(stream)
        self._s_in.wait_stream(stream)
        self._s_out.wait_stream(stream)
        for i in range(steps):
            b = i % 2
            st = self._sets[b]
            with torch.cuda.stream(self._s_in):
                if in_free[b] is not None:
                    self._s_in.wait_event(in_free[b])
                for n in self.e2e_in:
                    st[n].copy_(self.host[n], non_blocking=True)
                in_ready[b].record(self._s_in)
            stream.wait_event(in_ready[b])
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            self.buf.update(st)
            self.step()
            done = ev()
            done.record(stream)
            in_free[b] = done
            with torch.cuda.stream(self._s_out):
                self._s_out.wait_event(done)
                for n in self.e2e_out:
                    self._outs_host[b][n].copy_(st[n], non_blocking=True)
                out_ready[b].record(self._s_out)
            out_free[b] = out_ready[b]
            out_ready[b] = ev()
        stream.wait_stream(self._s_in)
        stream.wait_stream(self._s_out)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        self.e2e_mode = False
        self.e2e_last = self._outs_host[(steps - 1) % 2]
        self.buf.update(self._sets[0])
        return t0.elapsed_time(t1) / 1e3

    def e2e_check(self):
        """The host copy of the last pipelined step equals a fresh device-only step."""
        self.step()
        torch.cuda.synchronize(self.dev)
        return all(bool(torch.equal(self.buf[n].cpu(), self.e2e_last[n])) for n in self.e2e_out)

    def e2e_bytes(self):
        h2d = sum(self.host[n].numel() * self.host[n].element_size() for n in self.e2e_in)
        d2h = sum(self.buf[n].numel() * self.buf[n].element_size() for n in self.e2e_out)
        return h2d, d2h


def prefill_config(w):
    return {"workload": f"{w.name} prefill pass-KV: {w.num_seqs}x{w.seq_len} tokens, "
                        f"{w.num_q_heads}/{w.num_kv_heads} heads, d={w.head_dim}, cp={w.cp}",
            "seq_len": w.seq_len, "global_batch": w.num_seqs, "cp": w.cp,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "mode": "pass_kv"}


def line_config(w, ws, runner=None):
    """The `config` of a JSON line (the same for both arms)."""
    base = (prefill_config(w) if w.kind == "pass_kv" else
            runner.config() if runner is not None else
            {"workload": w.name, "global_batch": w.num_seqs, "cp": w.cp, "mode": w.kind})
    return dict(base, l2="flushed between timed steps (512 MB write)",
                parallelism=f"replicas x{ws} (logical CP shards on each GPU)")


class PrefillRunner(Runner):
    """pass-KV prefill: partition -> partial attention -> merge (or the fused launch)."""

    e2e_in = ("q", "k", "v", "cu")
    e2e_out = ("out",)
    e2e_note = ("throughput across steps: the inputs of step i+1 and the output of step i-1 "
                "are copied on two copy streams while step i computes (double-buffered sets)")

    def __init__(self, w, dev, cpa):
        super().__init__(dev, cpa)
        self.w = w
        lens = [w.seq_len] * w.num_seqs
        self.x = wl.prefill_inputs(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype, w.seed)
        self.lens = lens
        self.N = N = sum(lens)
        cp, Hq, d = w.cp, w.num_q_heads, w.head_dim
        self.buf = {
            "q": self.x["q"].to(dev), "k": self.x["k"].to(dev), "v": self.x["v"].to(dev),
            "cu": self.x["cu_seqlens"].to(dev),
            "part": torch.empty(cp, N, Hq, d, dtype=torch.float32, device=dev),
            "plse": torch.empty(cp, N, Hq, dtype=torch.float32, device=dev),
            "out": torch.empty(N, Hq, d, dtype=w.dtype, device=dev),
            "olse": torch.empty(N, Hq, dtype=torch.float32, device=dev),
            "perm": torch.empty(N, dtype=torch.int32, device=dev),
            "inv": torch.empty(N, dtype=torch.int32, device=dev),
            "so": torch.empty(cp + 1, dtype=torch.int32, device=dev),
            "cb": torch.empty(len(lens), 2 * cp + 1, dtype=torch.int32, device=dev),
        }
        self.flops = 4.0 * d * Hq * causal_pairs_pass_kv(lens)
        self.impl = cpa.CP_IMPL_AUTO
        self.fused = False

    def step(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        run_with_side_maps(
            self, lambda: cpa.cp_partition(b["cu"], w.cp, self.N, b["perm"], b["inv"], b["so"], b["cb"]),
            lambda: self._attention(ev))

    def _attention(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        if ev is not None:
            ev[0].record()
        if self.fused:  # every kv shard walked inside one item: final output, no partials
            cpa.cp_attn_prefill_fused(b["q"], b["cu"], w.cp, b["k"], b["v"],
                                      max_seqlen_q=max(self.lens), out=b["out"], out_lse=b["olse"],
                                      impl=self.impl)
            if ev is not None:
                ev[1].record()
            return
        cpa.cp_partial_attn_prefill(b["q"], b["cu"], w.cp, k=b["k"], v=b["v"],
                                    max_seqlen_q=max(self.lens), out=b["part"], lse=b["plse"],
                                    impl=self.impl)
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(b["part"], b["plse"], out=b["out"], out_lse=b["olse"])

    def merge_only(self):
        b = self.buf
        self.cpa.cp_lse_merge(b["part"], b["plse"], out=b["out"], out_lse=b["olse"])

    def merge_bytes(self):
        """Algorithmic bytes of one merge over the current partials: every partial LSE, the out
        rows of the non-empty partials, the merged output and its LSE."""
        b = self.buf
        P, R, H, d = b["part"].shape
        live = int(torch.isfinite(b["plse"]).sum().item())
        return P * R * H * 4 + live * d * 4 + R * H * (d * b["out"].element_size() + 4)

    @property
    def launches_per_step(self):
        return 2 if self.fused else 3

    def metric(self, seconds):
        return self.flops / seconds / 1e12

    def config(self):
        return prefill_config(self.w)


class PassQRunner(Runner):
    """chunked prefill (pass-Q): partition of the new tokens -> round-robin layout of the kv
    -> pass-Q partial attention over the paged cache -> merge.  End to end, each step also
    stores the new tokens' K/V into the paged cache (cp_kv_cache_write)."""

    e2e_in = ("q", "k_new", "v_new", "tables", "seq_lens", "cu_q", "cu_kv", "start")
    e2e_out = ("out",)
    e2e_note = ("throughput across steps (double-buffered sets, two copy streams); every step "
                "also writes its new tokens' K/V into the resident paged cache")

    def __init__(self, w, dev, cpa):
        super().__init__(dev, cpa)
        self.w = w
        self.x = x = wl.workload_inputs(w)
        B, cp, Hq, Hkv, d = w.num_seqs, w.cp, w.num_q_heads, w.num_kv_heads, w.head_dim
        self.N = N = B * w.q_len
        cu = [0]
        for L in x["seq_lens"].tolist():
            cu.append(cu[-1] + L)
        g = torch.Generator().manual_seed(w.seed + 500)
        self.buf = {
            "q": x["q"].to(dev), "kc": x["k_cache"].to(dev), "vc": x["v_cache"].to(dev),
            "tables": x["block_tables"].to(dev), "seq_lens": x["seq_lens"].to(dev),
            "cu_q": x["cu_seqlens_q"].to(dev),
            "cu_kv": torch.tensor(cu, dtype=torch.int32, device=dev),
            # new tokens' K/V of the end-to-end step (positions kv_len - q_len ..)
            "k_new": wl.normal((N, Hkv, d), w.dtype, g).to(dev),
            "v_new": wl.normal((N, Hkv, d), w.dtype, g).to(dev),
            "start": (x["seq_lens"] - w.q_len).to(dev),
            "part": torch.empty(cp, N, Hq, d, dtype=torch.float32, device=dev),
            "plse": torch.empty(cp, N, Hq, dtype=torch.float32, device=dev),
            "out": torch.empty(N, Hq, d, dtype=w.dtype, device=dev),
            "olse": torch.empty(N, Hq, dtype=torch.float32, device=dev),
            "local_lens": torch.empty(cp, B, dtype=torch.int32, device=dev),
            "perm": torch.empty(N, dtype=torch.int32, device=dev),
            "inv": torch.empty(N, dtype=torch.int32, device=dev),
            "so": torch.empty(cp + 1, dtype=torch.int32, device=dev),
            "cb": torch.empty(B, 2 * cp + 1, dtype=torch.int32, device=dev),
        }
        ctx = w.kv_len - w.q_len
        pairs = sum(ctx + i + 1 for i in range(w.q_len)) * B
        self.flops = 4.0 * d * Hq * pairs
        self.impl = cpa.CP_IMPL_AUTO
        self.fused = False
        # the fused form's tail-split workspace (0 bytes: every item runs whole)
        self.split_bytes = cpa.cp_prefill_fused_workspace_size(B, Hq, Hkv, d, cp, w.q_len)
        self.buf["fws"] = torch.empty(self.split_bytes, dtype=torch.uint8, device=dev)

    def step(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        if self.e2e_mode:  # the new tokens' K/V into their ranks' pages before attention
            cpa.cp_kv_cache_write(b["k_new"], b["v_new"], b["cu_q"], b["start"], b["kc"], b["vc"],
                                  b["tables"], w.cp, w.interleave)

        def maps():
            cpa.cp_partition(b["cu_q"], w.cp, self.N, b["perm"], b["inv"], b["so"], b["cb"])
            cpa.cp_kv_interleave_layout(b["cu_kv"], w.cp, w.interleave, 0, w.block_size,
                                        local_lens=b["local_lens"], want_slots=False)

        run_with_side_maps(self, maps, lambda: self._attention(ev))

    @property
    def launches_per_step(self):
        # fused: attention (+ the split tail's merge) ; else attention + merge; both + 2 maps
        return (3 + (self.split_bytes > 0)) if self.fused else 4

    def _attention(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        kw = dict(mode=cpa.CP_PASS_Q, k_cache=b["kc"], v_cache=b["vc"], block_tables=b["tables"],
                  seq_lens_kv=b["seq_lens"], interleave=w.interleave, max_seqlen_q=w.q_len,
                  impl=self.impl)
        if ev is not None:
            ev[0].record()
        if self.fused:  # every rank's resident pages walked inside one item: final output
            cpa.cp_attn_prefill_fused(b["q"], b["cu_q"], w.cp, out=b["out"], out_lse=b["olse"],
                                      workspace=b["fws"], **kw)
            if ev is not None:
                ev[1].record()
            return
        cpa.cp_partial_attn_prefill(b["q"], b["cu_q"], w.cp, out=b["part"], lse=b["plse"], **kw)
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(b["part"], b["plse"], out=b["out"], out_lse=b["olse"])

    def metric(self, seconds):
        return self.flops / seconds / 1e12

    def config(self):
        w = self.w
        return {"workload": f"chunked prefill pass-Q: {w.num_seqs} seqs x {w.q_len} new of "
                            f"{w.kv_len} kv, {w.num_q_heads}/{w.num_kv_heads} heads, d={w.head_dim}, "
                            f"paged bs={w.block_size}, cp={w.cp}, I={w.interleave}",
                "mode": "pass_q"}


class DecodeRunner(Runner):
    """decode: interleave layout -> per-rank split partials -> merge.  End to end, each step
    also stores the new token's K/V (position L-1) into the paged cache."""

    e2e_in = ("q", "k_new", "v_new", "seq_lens", "tables", "cu", "start", "cu_new")
    e2e_out = ("out",)
    e2e_note = ("throughput across steps (double-buffered sets, two copy streams); the paged "
                "cache stays resident, every step writes its new token's K/V into it")

    def __init__(self, w, dev, cpa):
        super().__init__(dev, cpa)
        self.w = w
        lens = wl.decode_lengths(w.num_seqs, w.min_len, w.max_len, w.len_seed).tolist()
        self.lens = lens
        caps = [wl.block_capacity(L, w.cp, w.interleave, w.block_size) for L in lens]
        tables, pool = wl.shuffled_block_tables(caps, w.cp, torch.Generator().manual_seed(w.table_seed))
        B, Hq, Hkv, d, cp = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cp
        g = torch.Generator(device=dev).manual_seed(w.seed)
        shape = (cp, pool, Hkv, w.block_size, d)
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        self.buf = {
            # kv values drawn on the device (same N(0,1) recipe; ~4.4 GB would take minutes on
            # the host), parity is checked on sampled sequences copied back
            "kc": torch.randn(shape, generator=g, device=dev, dtype=w.dtype),
            "vc": torch.randn(shape, generator=g, device=dev, dtype=w.dtype),
            "q": torch.randn(B, Hq, d, generator=g, device=dev, dtype=w.dtype),
            "k_new": torch.randn(B, Hkv, d, generator=g, device=dev, dtype=w.dtype),
            "v_new": torch.randn(B, Hkv, d, generator=g, device=dev, dtype=w.dtype),
            "tables": tables.to(dev),
            "seq_lens": torch.tensor(lens, dtype=torch.int32, device=dev),
            "start": torch.tensor([L - 1 for L in lens], dtype=torch.int32, device=dev),
            "cu_new": torch.arange(B + 1, dtype=torch.int32, device=dev),
            "cu": torch.tensor(cu, dtype=torch.int32, device=dev),
            "out": torch.empty(B, Hq, d, dtype=w.dtype, device=dev),
            "olse": torch.empty(B, Hq, dtype=torch.float32, device=dev),
            "local_lens": torch.empty(cp, B, dtype=torch.int32, device=dev),
        }
        self.ns, self.st = cpa.cp_decode_plan(B, Hkv, cp, w.interleave, w.block_size, max(lens))
        self._alloc_partials()
        self.fused = False  # two launches measured faster than the fused one
        el = torch.tensor([], dtype=w.dtype).element_size()
        pages = sum(-(-n // w.block_size) for L in lens
                    for n in [(L // (w.interleave * cp)) * w.interleave
                              + min(max(L % (w.interleave * cp) - r * w.interleave, 0), w.interleave)
                              for r in range(cp)])
        self.bytes = (sum(lens) * Hkv * d * 2 * el + 2 * B * Hq * d * el + pages * 4)
        self.pool = pool

    def _alloc_partials(self):
        w, dev = self.w, self.dev
        P = w.cp * self.ns
        B, Hq, Hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
        self.buf["part"] = torch.empty(P, B, Hq, d, dtype=torch.float32, device=dev)
        self.buf["plse"] = torch.empty(P, B, Hq, dtype=torch.float32, device=dev)
        self.buf["ws"] = torch.zeros(self.cpa.cp_decode_workspace_size(B, Hq, Hkv, d, w.cp, self.ns),
                                     dtype=torch.uint8, device=dev)

    def resplit(self, split_tokens):
        share = self.ns * self.st  # the planned split covers the largest rank share
        self.st = split_tokens
        self.ns = -(-share // split_tokens)
        self._alloc_partials()

    @property
    def launches_per_step(self):
        return 2 if self.fused else 3

    def step(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        if self.e2e_mode:  # the new token's K/V into its rank's page before attention
            cpa.cp_kv_cache_write(b["k_new"], b["v_new"], b["cu_new"], b["start"], b["kc"], b["vc"],
                                  b["tables"], w.cp, w.interleave)
        run_with_side_maps(
            self, lambda: cpa.cp_kv_interleave_layout(b["cu"], w.cp, w.interleave, 0, w.block_size,
                                                      local_lens=b["local_lens"], want_slots=False),
            lambda: self._attention(ev))

    def _attention(self, ev=None):
        cpa, w, b = self.cpa, self.w, self.buf
        if ev is not None:
            ev[0].record()
        if self.fused:  # partials + merge in one launch
            cpa.cp_decode_attention(b["q"], b["kc"], b["vc"], b["tables"], b["seq_lens"], w.cp,
                                    w.interleave, num_splits=self.ns, split_tokens=self.st,
                                    workspace=b["ws"], out=b["out"], out_lse=b["olse"])
            if ev is not None:
                ev[1].record()
            return
        cpa.cp_partial_attn_decode(b["q"], b["kc"], b["vc"], b["tables"], b["seq_lens"], w.cp,
                                   w.interleave, num_splits=self.ns, split_tokens=self.st,
                                   out=b["part"], lse=b["plse"])
        if ev is not None:
            ev[1].record()
        cpa.cp_lse_merge(b["part"], b["plse"], out=b["out"], out_lse=b["olse"])

    def metric(self, seconds):
        return self.bytes / seconds / 1e9

    def config(self):
        w = self.w
        return {"workload": f"decode: {w.num_seqs} seqs, ctx U[{w.min_len},{w.max_len}] "
                            f"(sum {sum(self.lens)}), {w.num_q_heads}/{w.num_kv_heads} heads, "
                            f"d={w.head_dim}, paged bs={w.block_size}, cp={w.cp}, I={w.interleave}",
                "splits": self.ns, "split_tokens": self.st}


def time_steps(runner, steps, warmup, flush, dev, stream, dominant=True, stretch_s=0.0, fn=None):
    """Per-step device time (CUDA events on the launching stream), L2 flushed between steps.
    `fn` (default runner.step) is the timed call; it records the dominant kernel's events."""
    fn = fn or runner.step
    for _ in range(warmup):
        flush.zero_()
        fn()
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
        if dominant:
            fn(dom[i])
        else:
            fn()
        ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    t1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dom_ms = [a.elapsed_time(b) for a, b in dom] if dominant else []
    return step_ms, dom_ms, (t0, t1)


# ------------------------------------------------------------------------------------- oracle

_INPUTS = {}


def _prefill_host_inputs(w):
    key = (w.name, w.num_seqs, w.seq_len, w.seed)
    if key not in _INPUTS:
        _INPUTS[key] = wl.prefill_inputs([w.seq_len] * w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                         w.head_dim, w.dtype, w.seed)
    return _INPUTS[key]


def sampled_rows(w, per_seq, seed, T):
    """Stratified query rows (global token rows) of every sequence: per_seq rows each."""
    from oracle import cp_oracle as orc
    bnd = orc.chunk_bounds(T, w.cp).tolist()
    rows = []
    for b in range(w.num_seqs):
        rows += [b * T + r for r in wl.sample_rows(T, bnd, per_seq, seed + b)]
    return rows


def oracle_pass_kv(w, per_seq, seed, x=None):
    """The float64 oracle (pass-KV partials + merge) on stratified query rows of the workload.
    Returns (causal flops of those rows, seconds, rows, (rows, O, LSE))."""
    from oracle import cp_oracle as orc
    x = x if x is not None else _prefill_host_inputs(w)
    rows = sampled_rows(w, per_seq, seed, w.seq_len)
    t = time.time()
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], w.cp,
                                1 / math.sqrt(w.head_dim), rows=rows)
    Om, Lm = orc.lse_merge(O, L)
    dt = time.time() - t
    flops = 4.0 * w.head_dim * w.num_q_heads * sum(r % w.seq_len + 1 for r in rows)
    return flops, dt, len(rows), (rows, Om, Lm)


def oracle_pass_q(w, x, per_seq, seed):
    """The float64 oracle (pass-Q partials + merge) on stratified new-query rows."""
    from oracle import cp_oracle as orc
    rows = sampled_rows(w, per_seq, seed, w.q_len)
    O, L = orc.pass_q_partials(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["cu_seqlens_q"], x["seq_lens"], w.cp, w.interleave,
                               w.block_size, 1 / math.sqrt(w.head_dim), rows=rows)
    Om, Lm = orc.lse_merge(O, L)
    return rows, Om, Lm


def oracle_decode(runner, seqs):
    """The float64 oracle (decode partials + merge) for the sampled sequences: their pages are
    copied back to the host into a compact pool (tables renumbered) first."""
    from oracle import cp_oracle as orc
    w, b = runner.w, runner.buf
    tables = b["tables"].cpu()
    cp = w.cp
    ids = [[int(p) for s in seqs for p in tables[r, s].tolist() if p >= 0] for r in range(cp)]
    n = max(len(x) for x in ids)
    shape = (cp, n) + tuple(b["kc"].shape[2:])
    kc = torch.zeros(shape, dtype=b["kc"].dtype)
    vc = torch.zeros(shape, dtype=b["vc"].dtype)
    new_tables = torch.full((cp, len(seqs), tables.shape[-1]), -1, dtype=torch.int32)
    for r in range(cp):
        idx = torch.tensor(ids[r], dtype=torch.long, device=b["kc"].device)
        kc[r, :len(ids[r])] = b["kc"][r].index_select(0, idx).cpu()
        vc[r, :len(ids[r])] = b["vc"][r].index_select(0, idx).cpu()
        remap = {p: i for i, p in enumerate(ids[r])}
        for j, s in enumerate(seqs):
            row = [remap[int(p)] for p in tables[r, s].tolist() if p >= 0]
            new_tables[r, j, :len(row)] = torch.tensor(row, dtype=torch.int32)
    q = b["q"].index_select(0, torch.tensor(seqs, device=b["q"].device)).cpu()
    lens = torch.tensor([runner.lens[s] for s in seqs], dtype=torch.int32)
    O, L = orc.decode_partials(q, kc, vc, new_tables, lens, cp, w.interleave, w.block_size,
                               1 / math.sqrt(w.head_dim))
    return orc.lse_merge(O, L)


def parity_block(out, lse, rows, Om, Lm, what):
    """Max errors of the GPU's merged output rows against the oracle's (same seeded inputs)."""
    import numpy as np
    idx = torch.as_tensor(rows, dtype=torch.long, device=out.device)
    o = out.index_select(0, idx).double().cpu().numpy()
    l = lse.index_select(0, idx).double().cpu().numpy()
    fin = np.isfinite(Lm)
    tol = 1e-2 + (2.0 ** -8 * np.abs(Om) if out.dtype == torch.bfloat16 else 0.0)
    err = np.abs(o - Om)
    lrel = np.abs(l[fin] - Lm[fin]) / np.abs(Lm[fin]).clip(1e-30)
    return {"rows": what, "max_abs_out": float(err.max()),
            "max_rel_lse": float(lrel.max()) if lrel.size else 0.0,
            "within_tolerance": bool((err <= tol).all() and
                                     (np.abs(l[fin] - Lm[fin]) <= 1e-3 * np.abs(Lm[fin]) + 1e-5).all()
                                     and np.array_equal(np.isfinite(l), fin)),
            "tolerance": "out 1e-2 + bf16 rounding 2^-8 |O|; lse 1e-3 relative + 1e-5"}


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


PREFILL_METRIC = "causal GQA prefill TFLOP/s (pass-KV partial attention + LSE merge)"


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = select_workload(args)
    if w.kind != "pass_kv":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle reference arm times "
                                                             "prefill workloads only"}))
        return 0
    per_seq = max(args.ref_rows // w.num_seqs, 4)
    _prefill_host_inputs(w)
    for i in range(args.warmup):
        oracle_pass_kv(w, max(per_seq // 8, 4), 9000 + i)
    tot_flops, tot_t, nrows = 0.0, 0.0, 0
    for i in range(args.steps):
        f, t, n, _ = oracle_pass_kv(w, per_seq, 9100 + i)
        tot_flops += f
        tot_t += t
        nrows += n
    val = tot_flops / tot_t / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": PREFILL_METRIC,
        "value": val, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(w, ws),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_seq} stratified query rows per sequence x all heads "
                                   f"per step ({nrows} rows total), float64 NumPy oracle"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def select_workload(args):
    w = wl.WORKLOADS[args.workload]
    if args.batch > 0:
        w = dataclasses.replace(w, num_seqs=args.batch)
    if args.cp > 0:
        w = dataclasses.replace(w, cp=args.cp)
    if args.interleave > 0:
        w = dataclasses.replace(w, interleave=args.interleave)
    if args.seed >= 0:
        w = dataclasses.replace(w, seed=args.seed)
    return w


def roofline(bound, kernel, work, dom_s, pk, traffic=None, algorithmic="", clk=None):
    """Dominant-kernel roofline.  A tensor-bound kernel is held against the burst bf16 peak,
    or against the sustained one when the clock samples of its own timed steps show the power
    cap engaged (as the sustained figure was measured)."""
    if bound == "tensor":
        capped = clk is not None and "sw_power_cap" in (clk.get("reasons") or [])
        peak, src = pk["bf16_sustained"] if capped else pk["bf16"]
        achieved = work / dom_s / 1e12
        unit = "TFLOP/s"
        psrc = (f"{src} bf16 dense (sustained: sw_power_cap during these steps)" if capped
                else f"{src} bf16 dense (burst)")
    else:
        peak, src = pk["hbm"]
        achieved = work / dom_s / 1e9
        unit, psrc = "GB/s", f"{src} HBM copy"
    return {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": psrc, "traffic": traffic,
            "algorithmic": algorithmic, "launch_ms": dom_s * 1e3}


def e2e_block(runner, steps, stream, ws, dev, unit, clocks=None):
    runner.e2e_run(3, stream)
    t0 = time.time()
    e2e_s = max_over_ranks(runner.e2e_run(steps, stream), ws, dev)
    t1 = time.time()
    if not runner.e2e_check():
        raise RuntimeError("end-to-end output differs from the device-only step")
    h2d, d2h = runner.e2e_bytes()
    e = {"value": runner.metric(e2e_s / steps) * ws, "unit": unit,
         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
         "pipelining": runner.e2e_note,
         "checked": "last host output == device-only step (bitwise)"}
    if clocks is not None:
        e["clocks"] = clocks.summary(t0, t1)
    return e


def traffic_key(runner):
    """The NCU_TRAFFIC record of a runner's dominant kernel in its current form."""
    kind = ("decode" if isinstance(runner, DecodeRunner) else
            "pass_q" if isinstance(runner, PassQRunner) else "prefill")
    return (kind + ("_fused" if runner.fused else ""), runner.w.name)


def prefill_kernel_name(runner):
    if isinstance(runner, PassQRunner):
        if runner.fused:
            return ("cp_attn_prefill_fused (pass-Q, paged, ranks merged in-kernel"
                    + ("; last wave's items split by rank range, then merged)" if runner.split_bytes
                       else ")"))
        return "cp_partial_attn_prefill (pass-Q, paged)"
    return ("cp_attn_prefill_fused (pass-KV, shards merged in-kernel)" if runner.fused
            else "cp_partial_attn_prefill (pass-KV)")


def measure_prefill_form(runner, fused, steps, flush, dev, stream, pk, clocks=None):
    """One prefill form (partials + merge, or the fused launch) of a runner: step value, the
    dominant kernel's roofline and the SM clocks sampled while it ran."""
    runner.fused = fused
    st, dm, win = time_steps(runner, steps, 3, flush, dev, stream)
    d_s = statistics.mean(dm) / 1e3
    clk = clocks.summary(*win) if clocks is not None else None
    e = {"value": runner.metric(statistics.mean(st) / 1e3), "unit": "TFLOP/s",
         "ms_per_step": statistics.mean(st),
         "roofline": roofline("tensor", prefill_kernel_name(runner), runner.flops, d_s, pk,
                              traffic=ncu_traffic(*traffic_key(runner)),
                              algorithmic=f"{runner.flops:.4e} causal FLOP per launch", clk=clk)}
    if clk is not None:
        e["clocks"] = clk
    return e


def settle(fn, dev, seconds):
    """Runs `fn` back to back for about `seconds`: after an idle host-side pause (the CPU oracle)
    a burst of GPU work met power-management transients (sw_power_cap with SM clocks at
    1.93-1.99 GHz for ~0.4 s), so each series of secondary measurements starts after a busy
    lead-in rather than straight after the pause."""
    t = time.time()
    while time.time() - t < seconds:
        for _ in range(4):
            fn()
        torch.cuda.synchronize(dev)


def secondaries(args, primary, w, dev, stream, flush, pk, ws, clocks=None):
    """Every other form and workload of the path, each with its dominant kernel's roofline and
    the SM clocks sampled over its timed steps."""
    sec = {}
    n = max(10, args.steps // 2)
    cpa = primary.cpa
    if isinstance(primary, PrefillRunner) and w.dtype == torch.bfloat16:
        primary.fused = True
        settle(primary.step, dev, 1.0)
        sec[f"{w.name}_prefill_fused"] = dict(
            measure_prefill_form(primary, True, n, flush, dev, stream, pk, clocks),
            config=primary.config())
        primary.fused = False
        # the LSE merge alone over the primary's partials
        primary.step()
        mb = primary.merge_bytes()
        st, _, win = time_steps(primary, n, 3, flush, dev, stream, dominant=False,
                                fn=primary.merge_only)
        m_s = statistics.mean(st) / 1e3
        sec["lse_merge"] = {"value": mb / m_s / 1e9, "unit": "GB/s", "config": primary.config(),
                            "roofline": roofline("hbm", "cp_lse_merge (merge_small_kernel)", mb, m_s, pk,
                                                 algorithmic=f"{mb:.4e} B per launch (every partial "
                                                             "LSE, non-empty partial rows, bf16 out + LSE)")}
        if clocks is not None:
            sec["lse_merge"]["clocks"] = clocks.summary(*win)
    if w.name != "full":
        fr = PrefillRunner(wl.WORKLOADS["full"], dev, cpa)
        settle(fr.step, dev, 0.5)
        for fused in (False, True):
            sec["full_prefill_fused" if fused else "full_prefill"] = dict(
                measure_prefill_form(fr, fused, n, flush, dev, stream, pk, clocks),
                config=fr.config())
        del fr
    if w.name != "chunked":
        qr = PassQRunner(wl.WORKLOADS["chunked"], dev, cpa)
        settle(qr.step, dev, 0.5)
        e = measure_prefill_form(qr, False, n, flush, dev, stream, pk, clocks)
        rows, Om, Lm = oracle_pass_q(qr.w, qr.x, 32, 4242)
        e["parity"] = parity_block(qr.buf["out"], qr.buf["olse"], rows, Om, Lm,
                                   f"{len(rows)} stratified new-query rows x all heads")
        e["e2e"] = e2e_block(qr, n, stream, ws, dev, "TFLOP/s", clocks)
        e["config"] = qr.config()
        sec["chunked_pass_q"] = e
        sec["chunked_pass_q_fused"] = dict(
            measure_prefill_form(qr, True, n, flush, dev, stream, pk, clocks), config=qr.config())
        del qr
    torch.cuda.empty_cache()
    dr = DecodeRunner(wl.WORKLOADS["decode"], dev, cpa)
    settle(dr.step, dev, 0.5)
    for fused in (False, True):
        dr.fused = fused
        ds, dd, win = time_steps(dr, max(10, args.steps // 5), 3, flush, dev, stream)
        d_s = statistics.mean(dd) / 1e3
        e = {"value": dr.metric(statistics.mean(ds) / 1e3), "unit": "GB/s", "config": dr.config(),
             "roofline": roofline("hbm", "cp_decode_attention (partials + merge, one launch)" if fused
                                  else "cp_partial_attn_decode", dr.bytes, d_s, pk,
                                  traffic=ncu_traffic(*traffic_key(dr)),
                                  algorithmic=f"{dr.bytes:.4e} B per launch (KV once + q + out + tables)")}
        if clocks is not None:
            e["clocks"] = clocks.summary(*win)
        seqs = [0, 1, 2, 3, 4, 5]
        Om, Lm = oracle_decode(dr, seqs)
        e["parity"] = parity_block(dr.buf["out"], dr.buf["olse"], seqs, Om, Lm,
                                   f"{len(seqs)} sequences x all heads")
        if not fused:
            e["e2e"] = e2e_block(dr, max(10, args.steps // 5), stream, ws, dev, "GB/s", clocks)
        sec["decode_fused" if fused else "decode"] = e
    del dr
    torch.cuda.empty_cache()
    return sec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long", choices=["long", "full", "tiny", "chunked", "decode"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=128,
                    help="reference arm: stratified query rows per step (over all sequences)")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="cpu baseline: stratified query rows per sequence (0: the workload's "
                         "sample size, all rows when it has none)")
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
    w = select_workload(args)
    runner = (DecodeRunner(w, dev, cpa) if w.kind == "decode" else
              PassQRunner(w, dev, cpa) if w.kind == "pass_q" else PrefillRunner(w, dev, cpa))
    if isinstance(runner, DecodeRunner):
        runner.fused = args.decode_fused
        if args.decode_split_tokens > 0:
            runner.resplit(args.decode_split_tokens)
    else:
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

    total_s = max_over_ranks(sum(step_ms) / 1e3, ws, dev)
    value = runner.metric(total_s / args.steps) * ws
    dom_s = statistics.mean(dom_ms) / 1e3

    if isinstance(runner, DecodeRunner):
        roof = roofline("hbm", "cp_decode_attention (partials + merge, one launch)" if runner.fused
                        else "cp_partial_attn_decode", runner.bytes, dom_s, pk,
                        traffic=ncu_traffic(*traffic_key(runner)),
                        algorithmic=f"{runner.bytes:.4e} B per launch (KV once + q + out + tables)")
        metric, unit = "decode KV-read GB/s (partial attention + LSE merge)", "GB/s"
    else:
        roof = roofline("tensor", prefill_kernel_name(runner), runner.flops, dom_s, pk,
                        traffic=ncu_traffic(*traffic_key(runner)),
                        algorithmic=f"{runner.flops:.4e} causal FLOP per launch", clk=clk)
        metric = (PREFILL_METRIC if isinstance(runner, PrefillRunner) and not runner.fused else
                  "causal GQA prefill TFLOP/s (" + prefill_kernel_name(runner) + ")")
        unit = "TFLOP/s"

    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": line_config(w, ws, runner),
            "roofline": roof, "clocks": clk,
            "gpu_launches": runner.launches_per_step * args.steps,
            "source_sha1": source_sha1()}

    # parity and the CPU baseline come from one oracle run over sampled rows of the workload
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and w.kind == "pass_kv":
        per_seq = args.cpu_rows or w.sample_rows or w.seq_len
        f, t, n, (rows, Om, Lm) = oracle_pass_kv(w, per_seq, 777, x=runner.x)
        if not runner.fused:
            runner.step()
            torch.cuda.synchronize(dev)
        line["parity"] = parity_block(runner.buf["out"], runner.buf["olse"], rows, Om, Lm,
                                      f"{n} stratified query rows x all heads" if n < runner.N
                                      else f"all {n} query rows x all heads")
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
                                "cpu_count": os.cpu_count(), "seconds": t,
                                "rows_per_s": n * w.num_q_heads / t, "kind": "oracle",
                                "sample": (f"all {n} query rows" if n >= runner.N
                                           else f"{n} stratified query rows ({per_seq} per sequence)")
                                          + f" x {w.num_q_heads} heads of the {w.name} workload, "
                                          f"float64 NumPy oracle, {t:.1f} s"}
    if not args.no_e2e and not (isinstance(runner, PrefillRunner) and runner.fused):
        settle(runner.step, dev, 1.0)  # after the oracle's host-side pause
        line["e2e"] = e2e_block(runner, args.steps, stream, ws, dev, unit, clocks)

    if not args.no_secondary and w.kind != "decode":
        line["secondary"] = secondaries(args, runner, w, dev, stream, flush, pk, ws, clocks)
    clocks.stop()

    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
