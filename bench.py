#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                    [--only] [--num-splits N]

One step is one call of the library's public entry point over one batch of
the workload (default: the GQA decode workload, B=8, Hq=32, Hkv=8, D=128,
KV cache padded to 8192 rows with per-batch lengths ~U[1024, 8192]). The
line also carries, in short form, the workloads beyond the five
configurations ("next_rows"), the decode split-count and warm-L2 sweeps
("decode_sweeps") and, last, all five configurations ("configs": step rate,
step and kernel times, the kernel's roofline fraction and DRAM traffic).

Timing: W untimed warm-up steps, then exactly K steps, each bracketed by
CUDA events on the launching stream; L2 is flushed (512 MB write) between
steps, outside the events. The main kernel is timed in a second pass of K
steps by events the library records right around it
(fa_set_main_kernel_events); they are kept out of the first pass, whose
step times they would inflate. Multi-GPU: one
process per GPU under torchrun; every rank runs its own replica of the
workload (weak scaling, no collective on the data path), the per-rank time
is max-reduced. With --impl reference the fp64 CPU oracle is timed instead
(rank 0 only) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "prefill attn TFLOP/s & decode KV-read GB/s on 1 GB300, as % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 * 1024 * 1024  # written, then half as much read: both above L2 (126 MB)
MAIN_KERNEL = {"decode": "decode_kernel", "prefill": "prefill_kernel"}
# the five configurations of the problem statement, by their workload names
CONFIGS = {"C1": "tiny_prefill", "C2": "gqa_decode", "C3": "long_decode",
           "C4": "causal_prefill", "C5": "gqa_masked_prefill"}
OTHER_WORKLOADS = ("long_decode", "causal_prefill", "gqa_masked_prefill", "tiny_prefill",
                   "window_prefill", "varlen_prefill", "d256_prefill", "paged_prefill",
                   "paged_decode", "d256_decode", "batch_decode", "gqa_decode")
# a forced split count (num_splits > 0) runs split_kernel instead of decode_kernel
SPLIT_KERNEL = "split_kernel"
KERNEL_SOURCE = {"decode_kernel": "attention_forward_qk_gb300/csrc/fa_decode.cu",
                 "split_kernel": "attention_forward_qk_gb300/csrc/fa_decode.cu",
                 "prefill_kernel": "attention_forward_qk_gb300/csrc/fa_prefill.cu"}


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def decode_lengths(w):
    """The per-batch valid lengths the workload generator draws (same seed, same order)."""
    import torch
    g = torch.Generator("cpu").manual_seed(w.seed)
    # the generator draws q, k, v first; replay those draws to reach the lengths
    for H, S in ((w.Hq, 1), (w.Hkv, w.S_kv), (w.Hkv, w.S_kv)):
        torch.randn((w.B, H, S, w.D), generator=g)
    if w.len_lo == w.len_hi:
        return [int(w.len_lo)] * w.B
    return [int(x) for x in torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=g)]


def prefill_pads(w):
    import torch
    if not w.max_pad:
        return None
    g = torch.Generator("cpu").manual_seed(w.seed)
    shp = {"BNSD": lambda H, S: (w.B, H, S, w.D), "BSND": lambda H, S: (w.B, S, H, w.D)}[w.layout]
    torch.randn(shp(w.Hq, w.S_q), generator=g)
    torch.randn(shp(w.Hkv, w.S_kv), generator=g)
    torch.randn(shp(w.Hkv, w.S_kv), generator=g)
    return [int(x) for x in torch.randint(0, w.max_pad + 1, (w.B,), generator=g)]


def work_units(w, lens=None, pads=None):
    """Algorithmic work of one step: decode -> bytes that must move (each valid
    K/V row once, q, out, lse); prefill -> FLOPs over unmasked (query, key)
    pairs only (4*D per pair: QK^T and PV)."""
    if w.kind == "decode":
        kv = 2 * 2 * w.D * w.Hkv * sum(lens)
        qo = 2 * 2 * w.B * w.Hq * w.D + 4 * w.B * w.Hq
        return {"step": kv + qo, "main": kv + 2 * w.B * w.Hq * w.D}
    S = w.S_q
    if w.packed:
        # lens: the packed sequences' lengths (q = kv)
        pairs = w.Hq * sum(L * (L + 1) // 2 if w.causal else L * L for L in lens)
        f = 4 * w.D * pairs
        return {"step": f, "main": f}
    if w.window is not None:
        wl, wr = w.window
        per_row = [min(S, i + wr + 1 if wr >= 0 else S) - max(0, i - wl if wl >= 0 else 0)
                   for i in range(S)]
        pairs = w.B * w.Hq * sum(per_row)
    elif w.causal and pads:
        pairs = w.Hq * sum(sum(min(i + 1, S - p) for i in range(S)) for p in pads)
    elif w.causal:
        pairs = w.B * w.Hq * S * (S + 1) // 2
    elif pads:
        pairs = w.Hq * S * sum(w.S_kv - p for p in pads)
    else:
        pairs = w.B * w.Hq * S * w.S_kv
    f = 4 * w.D * pairs
    return {"step": f, "main": f}


def traffic_from_profiles(kernel, workload):
    """Per-launch DRAM bytes of the main kernel from the committed ncu summary,
    or None when there is none or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    src = open(os.path.join(ROOT, KERNEL_SOURCE[kernel]), "rb").read()
    if hashlib.sha256(src).hexdigest() != h.group(1):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm

class Runner:
    """Inputs of one workload resident on the device and a callable step."""

    def __init__(self, w, dev, host_copy=False):
        import torch
        from attention_forward_qk_gb300 import fa as F
        self.w, self.dev, self.F = w, dev, F
        self.kind = w.kind
        # same seeded inputs as the parity tests
        x = workloads.make(w) if (host_copy or w.packed) else None
        self.cu = None
        if w.packed:
            self.lens = x["lengths"]
            self.cu = x["cu_seqlens"]
            self.pads = None
        elif w.kind == "decode":
            self.lens = x["lengths"] if x else decode_lengths(w)
            self.pads = None
        else:
            self.lens = None
            self.pads = x["pads"] if x else prefill_pads(w)
        self.units = work_units(w, self.lens, self.pads)
        if host_copy or w.packed:
            self.host = {k: (x[k].pin_memory() if host_copy else x[k]) for k in ("q", "k", "v")}
            if x.get("key_mask") is not None:
                self.host["key_mask"] = x["key_mask"].pin_memory()
            self.q = self.host["q"].to(dev)
            self.k = self.host["k"].to(dev)
            self.v = self.host["v"].to(dev)
            km = self.host.get("key_mask")
            self.km = km.to(dev) if km is not None else None
        else:
            g = torch.Generator(device=dev).manual_seed(w.seed)
            shp = (lambda H, S: (w.B, H, S, w.D)) if w.layout == "BNSD" else \
                (lambda H, S: (w.B, S, H, w.D))
            rnd = lambda s: torch.randn(s, generator=g, device=dev).to(torch.bfloat16)
            self.q, self.k, self.v = rnd(shp(w.Hq, w.S_q)), rnd(shp(w.Hkv, w.S_kv)), \
                rnd(shp(w.Hkv, w.S_kv))
            self.km = None
            if self.pads:
                km = torch.zeros(w.B, w.S_kv, dtype=torch.uint8)
                for b, p in enumerate(self.pads):
                    if p:
                        km[b, w.S_kv - p:] = 1
                self.km = km.to(dev)
        self.splits = 0  # fa_decode's num_splits (0 = one share per SM)
        self.table = None
        if w.block_size is not None:
            # scatter the cache into a pool of blocks in a seeded random order
            bs = w.block_size
            nb_seq = (w.S_kv + bs - 1) // bs
            perm = torch.randperm(w.B * nb_seq, generator=torch.Generator().manual_seed(w.seed))
            self.table = perm.view(w.B, nb_seq).to(torch.int32).to(dev)
            pool = lambda t: torch.empty(w.B * nb_seq, bs, w.Hkv, w.D, dtype=t.dtype, device=dev)
            kp, vp = pool(self.k), pool(self.v)
            kb = workloads.to_bnsd(self.k, w.layout)
            vb = workloads.to_bnsd(self.v, w.layout)
            idx = self.table.view(-1).long()
            kp[idx] = kb.reshape(w.B, w.Hkv, nb_seq, bs, w.D).permute(0, 2, 3, 1, 4) \
                .reshape(w.B * nb_seq, bs, w.Hkv, w.D)
            vp[idx] = vb.reshape(w.B, w.Hkv, nb_seq, bs, w.D).permute(0, 2, 3, 1, 4) \
                .reshape(w.B * nb_seq, bs, w.Hkv, w.D)
            self.k, self.v = kp, vp
            if host_copy:  # the end-to-end copies then move the pools
                self.host["k"] = kp.cpu().pin_memory()
                self.host["v"] = vp.cpu().pin_memory()
        self.out = torch.empty_like(self.q)
        lse_shape = (self.q.shape[0], w.Hq) if w.packed else (w.B, w.Hq, w.S_q)
        self.lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
        if w.packed:
            n = F.fa_forward_varlen_workspace_size(w.B, max(self.lens), max(self.lens), w.Hq,
                                                   w.Hkv, w.D)
        elif w.kind == "decode":
            n = F.fa_decode_workspace_size(w.B, w.S_kv, w.Hq, w.Hkv, w.D, 0)
        else:
            n = F.fa_forward_workspace_size(w.B, w.S_q, w.S_kv, w.Hq, w.Hkv, w.D)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def step(self):
        w, F = self.w, self.F
        if w.packed:
            F.fa_forward_varlen(self.q, self.k, self.v, self.cu, self.cu,
                                mask_mode="causal" if w.causal else None, scale=w.scale,
                                out=self.out, lse=self.lse, workspace=self.ws)
        elif self.table is not None and self.kind == "prefill":
            F.fa_forward_paged(self.q, self.k, self.v, self.table, w.block_size, w.S_kv,
                               kv_layout="PA_BBND", mask_mode="causal" if w.causal else None,
                               key_mask=self.km, scale=w.scale, layout=w.layout, out=self.out,
                               lse=self.lse, workspace=self.ws)
        elif self.kind == "decode" and self.table is not None:
            F.fa_decode_paged(self.q, self.k, self.v, self.table, w.block_size, self.lens,
                              scale=w.scale, num_splits=self.splits, out=self.out, lse=self.lse,
                              workspace=self.ws)
        elif self.kind == "decode":
            F.fa_decode(self.q, self.k, self.v, self.lens, scale=w.scale, layout=w.layout,
                        num_splits=self.splits, out=self.out, lse=self.lse, workspace=self.ws)
        elif w.window is not None:
            F.fa_forward_window(self.q, self.k, self.v, w.window[0], w.window[1],
                                key_mask=self.km, scale=w.scale, layout=w.layout, out=self.out,
                                lse=self.lse, workspace=self.ws)
        else:
            F.fa_forward(self.q, self.k, self.v, mask_mode="causal" if w.causal else None,
                         key_mask=self.km, scale=w.scale, layout=w.layout, out=self.out,
                         lse=self.lse, workspace=self.ws)

    def e2e_step(self, host_out, host_lse):
        """Pinned host inputs -> device, the call, results -> pinned host."""
        self.q.copy_(self.host["q"], non_blocking=True)
        self.k.copy_(self.host["k"], non_blocking=True)
        self.v.copy_(self.host["v"], non_blocking=True)
        if self.km is not None:
            self.km.copy_(self.host["key_mask"], non_blocking=True)
        self.step()
        host_out.copy_(self.out, non_blocking=True)
        host_lse.copy_(self.lse, non_blocking=True)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return self.out.numel() * self.out.element_size() + self.lse.numel() * 4


class L2Flush:
    """Evicts the step's inputs from L2 between steps: a 512 MB write, then a
    256 MB read, so that L2 is left holding clean lines of the flush buffers
    (the write-back of the flush's own dirty lines is not charged to the
    timed step)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.fill_(1.0)
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def sig(x, n=4):
    """x rounded to n significant digits (None stays None)."""
    return None if x is None else float(f"{x:.{n}g}")


def summary(r, full=False):
    """Short form of one workload's measurement for the JSON line: step rate,
    step and main-kernel times, the kernel's roofline fraction (and, for the
    five configurations, its achieved rate, bound and DRAM traffic)."""
    rf = r["roofline"]
    d = {"value": sig(r["value"]), "unit": r["unit"], "ms": sig(r["ms_per_step"]),
         "kernel_ms": sig(r["kernel_ms"]), "frac": sig(rf["frac"], 3)}
    if full:
        d.update({"kernel": rf["kernel"], "bound": rf["bound"], "achieved": sig(rf["achieved"]),
                  "traffic": rf["traffic"]})
    return d


def median(xs):
    s = sorted(xs)
    n = len(s)
    return (s[n // 2] + s[(n - 1) // 2]) / 2 if n else None


def time_steps(runner, steps, warmup, flush, fn=None, kernel=True):
    """Per-step CUDA-event times (ms) of `fn` (default runner.step) and of the
    main kernel inside it; L2 flushed before every step, outside the events.

    Two timed passes of `steps` steps each: the step times come from the
    first, where nothing but the two bracketing events is recorded; the main
    kernel's times from the second, where the library also records an event
    right before and after that kernel (an event between two launches breaks
    their programmatic overlap and costs stream time, so it would inflate the
    step time of the first pass). Launches are counted in the first pass."""
    import torch
    F = runner.F
    fn = fn or runner.step
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()

    def new_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in range(steps)]
        for e in evs:  # create the handles
            for x in e:
                x.record()
        torch.cuda.synchronize()
        return evs

    evs = new_events(2)
    l0 = F.fa_kernel_launch_count()
    for e in evs:
        flush()
        e[0].record()
        fn()
        e[1].record()
    torch.cuda.synchronize()
    launches = F.fa_kernel_launch_count() - l0
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    main_ms = []
    if kernel:
        kev = new_events(2)
        for e in kev:
            flush()
            F.fa_set_main_kernel_events(e[0], e[1])
            fn()
        F.fa_set_main_kernel_events(None, None)
        torch.cuda.synchronize()
        main_ms = [e[0].elapsed_time(e[1]) for e in kev]
    return step_ms, main_ms, launches


def roofline(kind, units_main, main_ms, peaks, peak_kind, workload, kernel=None):
    """`workload` names the committed profile (profiles/<kernel>_<workload>.md)
    whose DRAM bytes are the traffic."""
    kernel = kernel or MAIN_KERNEL[kind]
    if kind == "decode":
        achieved = units_main / (main_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                "traffic": traffic_from_profiles(kernel, workload)}
    achieved = units_main / (main_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_kind + " (burst)",
            "traffic": traffic_from_profiles(kernel, workload)}


def max_over_ranks(vals, world, device=None):
    """Each value's maximum over the ranks: the job takes as long as its
    slowest rank. A no-op on one rank."""
    if world == 1:
        return [float(v) for v in vals]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def value_of(kind, units, ms):
    if kind == "decode":
        return units / (ms * 1e-3) / 1e9, "GB/s"
    return units / (ms * 1e-3) / 1e12, "TFLOP/s"


def cpu_baseline(w, budget_s=12.0):
    """The fp64 oracle, as it stands, on this host's cores over a bounded
    sample of the workload: whole (batch) slices for decode, sampled query
    rows for prefill. Returns the same metric as the GPU line."""
    import numpy as np
    import oracle
    cores = len(os.sched_getaffinity(0))
    x = workloads.make(w)
    t0 = time.perf_counter()
    done_units, passes = 0.0, 0
    if w.kind == "decode":
        lens = x["lengths"]
        b = 0
        while time.perf_counter() - t0 < budget_s:
            sl = slice(b, b + 1)
            oracle.decode(x["q"][sl], x["k"][sl], x["v"][sl], lens[b:b + 1], scale=w.scale,
                          layout=w.layout)
            done_units += 2 * 2 * w.D * w.Hkv * lens[b]
            passes += 1
            b = (b + 1) % w.B
        el = time.perf_counter() - t0
        return {"value": done_units / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"{passes} single-batch decode passes of the workload "
                          f"({done_units / 1e6:.1f} MB of K/V), numpy fp64, {el:.1f} s"}
    rng = np.random.default_rng(0)
    pads = x.get("pads")
    rows_done = 0
    if w.packed:
        cu, lens = x["cu_seqlens"], x["lengths"]
        while time.perf_counter() - t0 < budget_s:
            b = passes % w.B
            L = lens[b]
            rows = sorted(rng.choice(L, size=min(16, L), replace=False).tolist())
            sl = slice(cu[b], cu[b + 1])
            oracle.attention(x["q"][sl][None], x["k"][sl][None], x["v"][sl][None], scale=w.scale,
                             layout="BSND", causal=w.causal, rows=rows)
            done_units += sum(4 * w.D * (i + 1 if w.causal else L) * w.Hq for i in rows)
            rows_done += len(rows)
            passes += 1
        el = time.perf_counter() - t0
        return {"value": done_units / el / 1e12, "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{rows_done} query rows x {w.Hq} heads in {passes} passes, numpy fp64, "
                          f"{el:.1f} s"}
    while time.perf_counter() - t0 < budget_s:
        rows = sorted(rng.choice(w.S_q, size=min(16, w.S_q), replace=False).tolist())
        bsl = slice(passes % w.B, passes % w.B + 1)
        km = x["key_mask"][bsl] if x["key_mask"] is not None else None
        oracle.attention(x["q"][bsl], x["k"][bsl], x["v"][bsl], scale=w.scale, layout=w.layout,
                         causal=w.causal, key_mask=km, rows=rows, window=w.window)
        p = pads[passes % w.B] if pads else 0
        for i in rows:
            if w.window is not None:
                wl, wr = w.window
                n = min(w.S_kv, i + wr + 1 if wr >= 0 else w.S_kv) - max(0, i - wl if wl >= 0 else 0)
            else:
                n = min(i + 1, w.S_kv - p) if w.causal else w.S_kv - p
            done_units += 4 * w.D * n * w.Hq
        rows_done += len(rows)
        passes += 1
    el = time.perf_counter() - t0
    return {"value": done_units / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows_done} query rows x {w.Hq} heads in {passes} passes, numpy fp64, "
                      f"{el:.1f} s"}


def F_ws_size(r, w, splits):
    """Workspace bytes of a decode call with `splits` pieces per sequence."""
    return r.F.fa_decode_workspace_size(w.B, w.S_kv, w.Hq, w.Hkv, w.D, splits)


def decode_sweeps(args, dev, flush, peaks, peak_kind):
    """The long decode workload with the K/V rows cut into a fixed number of
    pieces per sequence (num_splits 128 ... 1024) beside the default of one
    equal share per SM, and the GQA decode workload with L2 left warm between
    steps (its valid K/V rows, about 120 MB, then partly hit in the 126 MB L2)."""
    import torch
    out = {"C3_num_splits": {}, "C2_warm_l2": None}
    wl = workloads.WORKLOADS["long_decode"]
    r = Runner(wl, dev)
    for n in (0, 128, 256, 512, 1024):
        r.splits = n
        r.ws = torch.empty(r.F.fa_decode_workspace_size(wl.B, wl.S_kv, wl.Hq, wl.Hkv, wl.D, n),
                           dtype=torch.uint8, device=dev)
        r.step()
        s_ms, m_ms, _ = time_steps(r, args.steps, args.warmup, flush)
        o_ms, o_k = sum(s_ms) / len(s_ms), sum(m_ms) / len(m_ms)
        v, u = value_of("decode", r.units["step"], o_ms)
        rf = roofline("decode", r.units["main"], o_k, peaks, peak_kind, f"long_decode_s{n}",
                      kernel=SPLIT_KERNEL if n else None)
        # key "0": one equal share per SM (the default plan)
        out["C3_num_splits"][str(n)] = {"value": sig(v), "unit": u, "ms": sig(o_ms),
                                        "frac": sig(rf["frac"], 3), "kernel": rf["kernel"]}
    del r
    torch.cuda.empty_cache()
    wg = workloads.WORKLOADS["gqa_decode"]
    r = Runner(wg, dev)
    r.step()
    s_ms, m_ms, _ = time_steps(r, args.steps, args.warmup, lambda: None)
    o_ms, o_k = sum(s_ms) / len(s_ms), sum(m_ms) / len(m_ms)
    v, u = value_of("decode", r.units["step"], o_ms)
    rf = roofline("decode", r.units["main"], o_k, peaks, peak_kind, "gqa_decode")
    out["C2_warm_l2"] = {"value": sig(v), "unit": u, "ms": sig(o_ms),
                         "frac": sig(rf["frac"], 3), "l2": "not flushed between steps"}
    del r
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    w = workloads.WORKLOADS[args.workload]
    peaks, peak_kind = load_peaks()

    # the oracle baseline runs first, before any CUDA work (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from attention_forward_qk_gb300 import build as B
    B.build()
    flush = L2Flush(dev)
    main = Runner(w, dev, host_copy=True)
    if args.num_splits:
        # a forced split count: fixed-size pieces per sequence (split_kernel)
        main.splits = args.num_splits
        main.ws = torch.empty(F_ws_size(main, w, args.num_splits), dtype=torch.uint8, device=dev)

    sampler = ClockSampler(local)
    sampler.start()
    t_ramp = time.perf_counter()
    for _ in range(2000):  # bring clocks up before the timed region (untimed)
        if time.perf_counter() - t_ramp >= args.ramp_s:
            break
        main.step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms, main_ms, launches = time_steps(main, args.steps, args.warmup, flush)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()

    ms = sum(step_ms) / len(step_ms)
    kms = sum(main_ms) / len(main_ms)
    ms, kms, med_ms = max_over_ranks([ms, kms, median(step_ms)], world, dev)
    value, unit = value_of(w.kind, main.units["step"] * world, ms)

    # end to end through the public call: pinned host inputs in, results out
    host_out = torch.empty(main.out.shape, dtype=main.out.dtype, pin_memory=True)
    host_lse = torch.empty(main.lse.shape, dtype=torch.float32, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 20))
    e_ms, _, _ = time_steps(main, e2e_steps, 2, flush,
                            fn=lambda: main.e2e_step(host_out, host_lse), kernel=False)
    e2e_ms = sum(e_ms) / len(e_ms)
    (e2e_ms,) = max_over_ranks([e2e_ms], world, dev)
    e2e_val, _ = value_of(w.kind, main.units["step"] * world, e2e_ms)

    others, sweeps = {}, None
    if not args.only:
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            wo = workloads.WORKLOADS[name]
            r = Runner(wo, dev)
            r.step()
            s_ms, m_ms, _ = time_steps(r, args.steps, args.warmup, flush)
            o_ms = sum(s_ms) / len(s_ms)
            o_k = sum(m_ms) / len(m_ms)
            v, u = value_of(wo.kind, r.units["step"], o_ms)
            others[name] = {"value": v, "unit": u, "ms_per_step": o_ms,
                            "ms_per_step_median": median(s_ms), "kernel_ms": o_k,
                            "roofline": roofline(wo.kind, r.units["main"], o_k, peaks, peak_kind,
                                                 name)}
            del r
            torch.cuda.empty_cache()
        sweeps = decode_sweeps(args, dev, flush, peaks, peak_kind)

    if rank == 0:
        main_rf = roofline(w.kind, main.units["main"], kms, peaks, peak_kind,
                           w.name + (f"_s{args.num_splits}" if args.num_splits else ""),
                           kernel=SPLIT_KERNEL if args.num_splits else None)
        others[w.name] = {"value": value, "unit": unit, "ms_per_step": ms, "kernel_ms": kms,
                          "roofline": main_rf}
        line = {
            "metric": METRIC,
            "value": value,
            "unit": unit,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "ms_per_step_median": med_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16; stale cache rows are random bf16 bits)",
            "config": {"workload": w.name, "shape": w.note, "l2": "flushed between steps "
                       "(512 MB write then 256 MB read, outside the timed events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       **({"num_splits": args.num_splits} if args.num_splits else {})},
            "roofline": main_rf,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": unit, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": main.h2d_bytes(),
                    "d2h_bytes_per_step": main.d2h_bytes()},
            "gpu_launches": int(launches),
            "clocks": clocks,
        }
        if not args.only:
            # the workloads beyond the five configurations, then the sweeps, then
            # the five configurations last and compact (a reader that keeps only
            # the end of the line still sees all five)
            line["next_rows"] = {n: summary(others[n]) for n in OTHER_WORKLOADS
                                 if n in others and n not in CONFIGS.values()}
            line["decode_sweeps"] = sweeps
            line["configs"] = {f"{c} {n}": summary(others[n], full=True)
                               for c, n in CONFIGS.items() if n in others}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------ reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return  # rank 0 alone runs the CPU oracle
    w = workloads.WORKLOADS[args.workload]
    budget = max(0.5, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, budget_s=budget)
    vals = [cpu_baseline(w, budget_s=budget) for _ in range(args.steps)]
    value = statistics.mean(v["value"] for v in vals)
    unit = vals[0]["unit"]
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": budget * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": w.name, "shape": w.note},
        "cpu_baseline": {"value": value, "unit": unit, "cores": vals[0]["cores"],
                         "kind": "oracle", "sample": f"each step: {vals[0]['sample']}"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gqa_decode", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ramp-s", type=float, default=0.5,
                    help="untimed steps before the timed region, in seconds (clock ramp)")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="decode workloads: a forced number of K/V pieces per sequence "
                         "(0: one equal share per SM)")
    ap.add_argument("--oracle-all", action="store_true",
                    help="time the fp64 oracle on the five configurations (host cores only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.num_splits < 0 or (args.num_splits and
                               workloads.WORKLOADS[args.workload].kind != "decode"):
        ap.error("--num-splits takes a non-negative count and a decode workload")
    if args.num_splits and workloads.WORKLOADS[args.workload].block_size is not None:
        ap.error("--num-splits: the paged workload runs the default plan only")
    if args.oracle_all:
        # the oracle's own throughput on each configuration, a bounded sample
        # each (whole decode passes; sampled query rows for prefill)
        for name in ("tiny_prefill", "gqa_decode", "long_decode", "causal_prefill",
                     "gqa_masked_prefill"):
            r = cpu_baseline(workloads.WORKLOADS[name], budget_s=10.0)
            print(json.dumps({"workload": name, **r}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
