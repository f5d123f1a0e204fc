#!/usr/bin/env python3
"""Throughput of the context-parallel attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--mode fused|stepwise]
    python bench.py --impl reference ...      # the float64 CPU oracle on the host cores

One step = one cp_attention_fwd over the workload's resident synthetic inputs
(every row of the hot path: shard table, regroups when Ulysses is on, the
block-attention lap with its LSE merges). The K timed steps run back to back
between one pair of CUDA events, rotating over three seeded input sets that
together exceed the L2 cache (so no step finds its inputs there); the
secondary measurements flush L2 (a 512 MB write) between timed launches,
outside their events. With N > 1 (torchrun), every rank runs its own
independent problem on its own GPU (weak scaling, no data-path collective);
the time is the max over ranks. Clocks, power and clock-event reasons are
sampled inside each timed region through NVML about every millisecond
(nvidia-smi at 100 ms where NVML does not load).

Prints one JSON line (rank 0).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "context-parallel attention fwd TFLOP/s and % bf16 tensor peak on 1 GB300"
UNIT = "TFLOP/s"
E2E_HEAD_CHUNKS = 5  # head chunks of the host-buffer call
N_SETS = 3           # input sets the timed steps rotate over (together larger than L2)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_fwd_tc_flux_ring4.md")
TC_KERNEL_SOURCE = os.path.join(ROOT, "context_attention_dits_gb300", "csrc", "attn_tc.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="flux_ring4")
    ap.add_argument("--mode", default="fused", choices=["fused", "stepwise"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the per-kernel HBM measurements and the other workloads")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """Rank 0's ring lap (attention per block + LSE merge) for `rows` query rows of `heads` heads."""

    def __init__(self, w, q, k, v, rows, heads):
        import numpy as np
        import oracle
        self.oracle, self.w = oracle, w
        self.table = oracle.ring_shard_table(w.S, w.ring_degree, w.uneven_ok)
        off0 = self.table[0][0]
        hs = list(range(heads))
        self.q = q[:, off0:off0 + rows][:, :, hs].float().numpy().astype(np.float64)
        self.k = k[:, :, hs].float().numpy().astype(np.float64)
        self.v = v[:, :, hs].float().numpy().astype(np.float64)
        self.rows, self.heads = rows, heads
        self.flops = 4 * w.B * heads * rows * w.S * w.D

    def run(self):
        o = self.oracle
        acc = None
        R = len(self.table)
        for t in range(R):
            off, ln = self.table[(0 - t) % R]
            part = o.attention(self.q, self.k[:, off:off + ln], self.v[:, off:off + ln], self.w.scale)
            acc = part if acc is None else o.lse_merge(*acc, *part)
        return acc

    def describe(self):
        return (f"ring lap of rank 0 for {self.rows} query rows x {self.heads} heads x B={self.w.B} against all "
                f"{self.w.S} keys ({len(self.table)} blocks), float64 numpy")


def sized_sample(w, q, k, v, budget_s, heads_max):
    """Grow the sample until one run takes about budget_s seconds."""
    rows, heads = 16, 1
    while True:
        s = OracleSample(w, q, k, v, rows, heads)
        t0 = time.perf_counter()
        s.run()
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or (rows >= w.S // w.ring_degree and heads >= heads_max):
            return s, dt
        grow = max(1.5, min(8.0, budget_s * 0.7 / max(dt, 1e-4)))
        if rows < w.S // w.ring_degree:
            rows = min(w.S // w.ring_degree, int(rows * grow) + 1)
        else:
            heads = min(heads_max, int(heads * grow) + 1)


def cpu_baseline(w, q, k, v, budget_s=12.0):
    s, _ = sized_sample(w, q, k, v, budget_s / 3, w.H)
    reps, t0 = 0, time.perf_counter()
    while True:
        s.run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s * 0.8:
            break
    return {"value": s.flops * reps / el / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": s.describe(), "seconds": round(el, 3)}


# ---------------------------------------------------------------------------
# secondary lines: the HBM-bound kernels and the other workloads
# ---------------------------------------------------------------------------
def _time_events(fn, flush, stream, reps):
    """Mean CUDA-event time (ms) of fn over reps runs, L2 flushed before each (outside the events)."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(float(i))
        st[i].record(stream)
        fn()
        en[i].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(st, en)) / reps


def _time_batch(fns, flush, stream, rounds):
    """CUDA-event time (ms) per launch of the launch list fns run back to back, rounds times, L2
    flushed once before each round (outside the events). The operands of fns together exceed L2, so
    every launch reads from HBM; back-to-back launches overlap their launch latency, as the
    launches of a stepwise lap do."""
    import torch
    for f in fns:
        f()
    torch.cuda.synchronize()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(rounds)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(rounds)]
    for i in range(rounds):
        flush.fill_(float(i))
        st[i].record(stream)
        for f in fns:
            f()
        en[i].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(st, en)) / (rounds * len(fns))


def secondary(cpa, dev, flush, stream, peaks, clocks=None):
    """Achieved bandwidth of the merge and regroup kernels (algorithmic bytes / event time) and the
    throughput of cp_attention_fwd on the other workloads. Every line carries the clock summary of its
    own timed window."""
    import torch
    from synth import WORKLOADS, make_merge_operands, make_qkv
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {}
    win = {"t0": time.time()}

    def opened():
        torch.cuda.synchronize()
        win["t0"] = time.time()

    def closed(name):
        torch.cuda.synchronize()
        if clocks is not None and name in res:
            res[name]["clocks"] = clocks.summary((win["t0"], time.time()))
        win["t0"] = time.time()

    def bw(name, nbytes, ms_single, ms_batch, note):
        res[name] = {"bytes_per_launch": nbytes, "single_launch": {"ms": ms_single, "GB_s": nbytes / ms_single / 1e6,
                                                                   "frac_of_hbm": nbytes / ms_single / 1e6 / hbm},
                     "back_to_back": {"ms": ms_batch, "GB_s": nbytes / ms_batch / 1e6,
                                      "frac_of_hbm": nbytes / ms_batch / 1e6 / hbm},
                     "note": note}
        closed(name)

    def fwd_line(name, w, ms, launches, **extra):
        tf = w.flops / (ms * 1e-3) / 1e12
        res[name] = {"TFLOP_s": tf, "ms": ms, "frac_of_bf16_peak": tf / bf16, "launches": launches, **extra}
        closed(name)

    # LSE merge at the shape the stepwise FLUX ring-4 lap launches: one ring step's partial of all four
    # simulated ranks, [1,4608,24,128] fp32 + lse [1,24,4608] (171 MB); the lap runs three of them,
    # each after that step's attention launch
    opened()
    sets = [[t.to(dev) for t in make_merge_operands(1, 24, 4608, 128, seed=15 + i)] for i in range(3)]
    nbytes = 12 * sets[0][0].numel() + 12 * sets[0][1].numel()
    fns = [lambda o=o: cpa.cp_lse_merge(o[0], o[1], o[2], o[3], stream=stream) for o in sets]
    bw("lse_merge_flux_ring4_lap_step", nbytes, _time_events(fns[0], flush, stream, 20),
       _time_batch(fns, flush, stream, 5), "the launched shape; back_to_back: the lap's three merges")
    del sets, fns

    # LSE merge of one FLUX ring-4 rank-step partial: [1,1152,24,128] fp32 + lse [1,24,1152];
    # one rank's share of a lap step's merge. Eight operand sets (342 MB) rotate through the batch.
    B, S, H, D = 1, 1152, 24, 128
    opened()
    sets = [[t.to(dev) for t in make_merge_operands(B, H, S, D, seed=5 + i)] for i in range(8)]
    nbytes = 12 * sets[0][0].numel() + 12 * sets[0][1].numel()
    fns = [lambda o=o: cpa.cp_lse_merge(o[0], o[1], o[2], o[3], stream=stream) for o in sets]
    bw("lse_merge_flux_ring4_step", nbytes, _time_events(fns[0], flush, stream, 30),
       _time_batch(fns * 3, flush, stream, 5), "one rank-step merge; back_to_back: 24 merges over 8 operand sets")
    del sets, fns

    # the same merge at the unified video step shape (R=2 x U=4, S=32768: one step's partial of all
    # four head groups, [4, 32768, 6, 128] fp32, 402 MB), as the stepwise lap of that workload runs it
    oa, la, ob, lb = (t.to(dev) for t in make_merge_operands(4, 6, 32768, 128, seed=9))
    nbytes = 12 * oa.numel() + 12 * la.numel()
    opened()
    ms = _time_events(lambda: cpa.cp_lse_merge(oa, la, ob, lb, stream=stream), flush, stream, 10)
    res["lse_merge_video_unified_step"] = {"bytes_per_launch": nbytes, "single_launch": {
        "ms": ms, "GB_s": nbytes / ms / 1e6, "frac_of_hbm": nbytes / ms / 1e6 / hbm}}
    closed("lse_merge_video_unified_step")
    del oa, la, ob, lb

    # Ulysses regroups of FLUX Ulysses-4: q, k, v (bf16) seq->head; out (fp32) head->seq
    U, S, H, D = 4, 4608, 24, 128
    xs = [torch.randn((U, 1, S // U, H, D), device=dev).to(torch.bfloat16) for _ in range(6)]
    ys = [torch.empty((U, 1, S, H // U, D), device=dev, dtype=torch.bfloat16) for _ in range(6)]
    nbytes = 2 * xs[0].numel() * 2
    opened()
    fns = [lambda x=x, y=y: cpa.cp_ulysses_seq2head(x, y, stream=stream) for x, y in zip(xs, ys)]
    bw("seq2head_flux_ulysses4_bf16", nbytes, _time_events(fns[0], flush, stream, 30),
       _time_batch(fns * 2, flush, stream, 5), "one tensor; back_to_back: 12 regroups over 6 tensor pairs")
    del xs, ys, fns
    xs = [torch.randn((U, 1, S, H // U, D), device=dev) for _ in range(3)]
    ys = [torch.empty((U, 1, S // U, H, D), device=dev) for _ in range(3)]
    nbytes = 2 * xs[0].numel() * 4
    opened()
    fns = [lambda x=x, y=y: cpa.cp_ulysses_head2seq(x, y, stream=stream) for x, y in zip(xs, ys)]
    bw("head2seq_flux_ulysses4_f32", nbytes, _time_events(fns[0], flush, stream, 30),
       _time_batch(fns * 4, flush, stream, 5), "the fp32 output; back_to_back: 12 regroups over 3 tensor pairs")
    del xs, ys, fns
    # a Ulysses-4 regroup at video length: q (bf16) 4 x [1, 8192, 24, 128] -> 4 x [1, 32768, 6, 128]
    # (201 MB each way)
    x = torch.randn((1, 32768, 24, 128), device=dev).to(torch.bfloat16)
    y = torch.empty((4, 1, 32768, 6, 128), device=dev, dtype=torch.bfloat16)
    xr = x.view(1, 4, 8192, 24, 128).permute(1, 0, 2, 3, 4).contiguous()  # four 8192-token rank shards
    nbytes = 2 * x.numel() * 2
    opened()
    ms = _time_events(lambda: cpa.cp_ulysses_seq2head(xr.view(4, 1, 8192, 24, 128), y.view(4, 1, 32768, 6, 128),
                                                       stream=stream), flush, stream, 10)
    res["seq2head_32768tok_ulysses4_bf16"] = {"bytes_per_launch": nbytes, "single_launch": {
        "ms": ms, "GB_s": nbytes / ms / 1e6, "frac_of_hbm": nbytes / ms / 1e6 / hbm}}
    closed("seq2head_32768tok_ulysses4_bf16")
    del x, y, xr

    # the stepwise FLUX ring-4 lap as a whole (one attention launch per ring step over all ranks, fp32
    # partials, the merge after each step but the first), next to the fused lap of the same inputs
    w = WORKLOADS["flux_ring4"]
    q, k, v = (t.to(dev) for t in make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult))
    out = torch.empty((w.B, w.S, w.H, w.D), device=dev)
    lse = torch.empty((w.B, w.H, w.S), device=dev)
    for mode in ("stepwise", "fused"):
        wsb = cpa.cp_attention_workspace_size(w.B, w.H, w.S, w.D, w.ring_degree, 1, q.dtype, mode)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        opened()
        ms = _time_events(lambda: cpa.cp_attention_fwd(q, k, v, out, lse, w.scale, w.ring_degree, 1, False,
                                                        workspace=ws, mode=mode, stream=stream), flush, stream, 20)
        fwd_line(f"flux_ring4_{mode}", w, ms,
                 cpa.cp_attention_launch_count(w.B, w.H, w.S, w.D, w.ring_degree, 1, q.dtype, mode),
                 lap_mode=mode)
        del ws
    step_part = (w.B * w.S * w.H * w.D + w.B * w.H * w.S) * 4  # one step's fp32 partial (out + lse)
    extra_bytes = (w.ring_degree - 1) * 4 * step_part  # per later step: partial written, merge reads 2, writes 1
    extra_ms = res["flux_ring4_stepwise"]["ms"] - res["flux_ring4_fused"]["ms"]
    res["flux_ring4_stepwise"]["extra_vs_fused"] = {
        "ms": extra_ms, "algorithmic_bytes": extra_bytes,
        "GB_s": extra_bytes / extra_ms / 1e6 if extra_ms > 0 else None,
        "frac_of_hbm": extra_bytes / extra_ms / 1e6 / hbm if extra_ms > 0 else None,
        "note": "the partials' fp32 write and the merges' reads and write, over the stepwise lap's extra time"}
    del q, k, v, out, lse

    # cp_attention_fwd on the other workloads (fused lap), inputs resident
    for name in ("flux_ulysses4", "ring_anything3", "video_unified", "flux1008_ulysses_anything4",
                 "ulysses_anything5_heads"):
        w = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult))
        out = torch.empty((w.B, w.S, w.H, w.D), device=dev)
        lse = torch.empty((w.B, w.H, w.S), device=dev)
        wsb = cpa.cp_attention_workspace_size(w.B, w.H, w.S, w.D, w.ring_degree, w.ulysses_degree, q.dtype, "fused")
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        opened()
        ms = _time_events(lambda: cpa.cp_attention_fwd(q, k, v, out, lse, w.scale, w.ring_degree,
                                                        w.ulysses_degree, w.uneven_ok, workspace=ws,
                                                        mode="fused", stream=stream),
                          flush, stream, 5 if name == "video_unified" else 20)
        fwd_line(name, w, ms, cpa.cp_attention_launch_count(w.B, w.H, w.S, w.D, w.ring_degree,
                                                             w.ulysses_degree, q.dtype, "fused"))
        if name == "flux_ulysses4":
            # the same attention launch alone, on head-grouped copies [U*B, S, H/U, D]: what the call adds on
            # top is the cost of its regroups (q, k, v seq->head; out, lse head->seq)
            U, Hg = w.ulysses_degree, w.H // w.ulysses_degree
            qh, kh, vh = (t.view(w.B, w.S, U, Hg, w.D).permute(2, 0, 1, 3, 4).reshape(U * w.B, w.S, Hg, w.D)
                          .contiguous() for t in (q, k, v))
            oh = torch.empty((U * w.B, w.S, Hg, w.D), device=dev)
            lh = torch.empty((U * w.B, Hg, w.S), device=dev)
            opened()
            ms_attn = _time_events(lambda: cpa.cp_block_attn_fwd(qh, kh, vh, oh, lh, w.scale, stream=stream),
                                   flush, stream, 20)
            rg_bytes = 2 * 3 * q.numel() * q.element_size() + 2 * (out.numel() + lse.numel()) * 4
            rg_ms = ms - ms_attn
            res[name]["regroup_cost"] = {
                "attention_only_ms": ms_attn, "regroups_ms": rg_ms, "regroup_bytes": rg_bytes,
                "GB_s": rg_bytes / rg_ms / 1e6 if rg_ms > 0 else None,
                "frac_of_hbm": rg_bytes / rg_ms / 1e6 / hbm if rg_ms > 0 else None,
                "note": "call time minus the attention launch alone; regroups move 2 x (q, k, v, out, lse)"}
            closed(name)
            del qh, kh, vh, oh, lh
        del q, k, v, out, lse, ws
    # key-padding mask: FLUX ring 4 with text keys 300..511 masked (FLOPs counted dense, as unmasked)
    w = WORKLOADS["flux_ring4"]
    q, k, v = (t.to(dev) for t in make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult))
    out = torch.empty((w.B, w.S, w.H, w.D), device=dev)
    lse = torch.empty((w.B, w.H, w.S), device=dev)
    km = torch.ones((w.B, w.S), dtype=torch.bool, device=dev)
    km[:, 300:512] = False
    opened()
    ms = _time_events(lambda: cpa.cp_attention_fwd(q, k, v, out, lse, w.scale, w.ring_degree, 1, False,
                                                    mode="fused", stream=stream, key_mask=km), flush, stream, 20)
    fwd_line("flux_ring4_text_padding_mask", w, ms, 1, note="keys 300..511 masked; FLOPs counted as unmasked")
    del q, k, v, out, lse, km

    # backward of the FLUX ring-4 and Ulysses-4 forwards: algorithmic FLOPs are 2.5x the forward's
    # (five S x S x D products per head: s recomputed, dp, dv, dq, dk); bf16 runs on the tensor cores
    from synth import make_dout
    for name, R, U in (("flux_ring4_bwd", 4, 1), ("flux_ulysses4_bwd", 1, 4)):
        w = WORKLOADS["flux_ring4"]
        q, k, v = (t.to(dev) for t in make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed))
        dout = make_dout(w.B, w.S, w.H, w.D, w.dtype, w.seed).to(dev)
        out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.float32, device=dev)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        cpa.cp_attention_fwd(q, k, v, out, lse, w.scale, R, U, stream=stream)
        grads = [torch.empty_like(out) for _ in range(3)]
        ws = torch.empty(max(1, cpa.cp_attention_bwd_workspace_size(w.B, w.H, w.S, w.D, R, U, q.dtype)),
                         dtype=torch.uint8, device=dev)
        opened()
        ms = _time_events(lambda: cpa.cp_attention_bwd(q, k, v, out, dout, lse, *grads, w.scale, R, U,
                                                       workspace=ws, stream=stream), flush, stream, 10)
        tf = 2.5 * w.flops / (ms * 1e-3) / 1e12
        res[name] = {"TFLOP_s": tf, "ms": ms, "frac_of_bf16_peak": tf / bf16,
                     "launches": cpa.cp_attention_bwd_launch_count(w.B, w.H, w.S, w.D, R, U, q.dtype),
                     "note": "tensor-core backward (dk/dv and dq kernels); FLOPs = 2.5 x forward"}
        closed(name)
        del q, k, v, dout, out, lse, grads, ws
    if cpa.cp_check_device_status() != 0:
        raise RuntimeError("device status after the secondary measurements")
    return res


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples, self.proc, self.thread, self.window = [], None, None, None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, window=None):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        t0, t1 = window or self.window or (0, float("inf"))
        inside = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not inside:  # a short timed region: take the samples nearest to it
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((num(p[2]) or 0.0) for p in inside)}


class NvmlClockSampler(ClockSampler):
    """The same record through NVML (the driver's libnvidia-ml; read-only queries), polled about every
    millisecond on a thread, so that a timed region of a few milliseconds still holds samples. Reason
    bits are NVML's clock-event reasons."""
    REASON_BITS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"), (0x20, "sw_thermal_slowdown"),
                   (0x4, "sw_power_cap"))

    def __init__(self, gpu_uuid):  # noqa: super().__init__ would start nvidia-smi
        import ctypes
        self.samples, self.proc, self.window, self.stopped = [], None, None, False
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib, self.c = lib, ctypes
        self.handle = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(str(gpu_uuid).encode(), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle for " + str(gpu_uuid))
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()

    def _poll(self):
        c = self.c
        sm, mx, mw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        while not self.stopped:
            ok = (self.lib.nvmlDeviceGetClockInfo(self.handle, 1, c.byref(sm)) == 0 and
                  self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, c.byref(mx)) == 0 and
                  self.lib.nvmlDeviceGetPowerUsage(self.handle, c.byref(mw)) == 0 and
                  self.reasons_fn(self.handle, c.byref(rs)) == 0)
            if ok:
                flags = ["Active" if rs.value & bit else "Not Active" for bit, _ in self.REASON_BITS]
                self.samples.append((time.time(), [str(sm.value), str(mx.value), str(mw.value / 1000.0)] + flags))
            time.sleep(0.001)

    def stop(self):
        self.stopped = True
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, window=None):
        # the window itself (samples are dense), else the sample nearest to it
        t0, t1 = window or self.window or (0, float("inf"))
        if self.samples and not any(t0 <= t <= t1 for t, _ in self.samples):
            return super().summary(window)
        saved = self.samples
        self.samples = [(t, p) for t, p in saved if t0 <= t <= t1]
        try:
            out = super().summary((t0 - 1.0, t1 + 1.0))
        finally:
            self.samples = saved
        out["source"] = "nvml, ~1 ms"
        return out


def clock_sampler(gpu_id):
    """NVML polling where the driver library loads, else nvidia-smi at 100 ms."""
    try:
        return NvmlClockSampler(gpu_id)
    except (OSError, AttributeError):
        return ClockSampler(gpu_id)


# ---------------------------------------------------------------------------
# traffic of the dominant kernel from the committed ncu summary
# ---------------------------------------------------------------------------
def profiled_traffic(workload, mode):
    if workload != "flux_ring4" or mode != "fused" or not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_tr):
        return None
    sha = hashlib.sha256(open(TC_KERNEL_SOURCE, "rb").read()).hexdigest()
    return float(m_tr.group(1)) if sha == m_sha.group(1) else None


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def reduce_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, w, world, rank):
    if rank != 0:
        return None
    from synth import make_qkv
    q, k, v = make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult)
    per_step = max(0.05, 90.0 / max(1, args.steps + args.warmup))
    s, _ = sized_sample(w, q, k, v, per_step, 1)
    for _ in range(args.warmup):
        s.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.run()
    el = time.perf_counter() - t0
    val = s.flops * args.steps / el / 1e12
    line = {"metric": METRIC, "value": val, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, args.mode),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": s.describe()},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    return line


def set_bytes_mb(w):
    """MB of one input set (q, k, v) of workload w."""
    return 3 * w.B * w.S * w.H * w.D * (2 if w.dtype == "bf16" else 4) / 1e6


def config_of(w, mode):
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "qkv_dtype": w.dtype,
            "ring_degree": w.ring_degree, "ulysses_degree": w.ulysses_degree, "uneven_ok": w.uneven_ok,
            "q_mult": w.q_mult, "lap_mode": mode, "scale": "1/sqrt(D)",
            "inputs": f"seeded N(0,1) (seed {w.seed}), resident in HBM",
            "l2": f"timed steps back to back over {N_SETS} rotating input sets ({N_SETS} x {set_bytes_mb(w):.0f} MB, "
                  f"larger than the 129 MB L2); no flush",
            "parallelism": f"simulated ring{w.ring_degree} x ulysses{w.ulysses_degree} on one GPU"}


def run_ours(args, w, world, rank, local):
    import numpy as np
    import torch

    import context_attention_dits_gb300 as cpa
    from synth import make_qkv

    dev = torch.device("cuda", torch.cuda.current_device())
    q_h, k_h, v_h = make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    # the timed steps rotate over N_SETS input sets (the first is the one above), so that their inputs
    # together exceed the L2 cache and no step finds the previous step's inputs there
    sets = [(q, k, v)] + [tuple(t.to(dev) for t in make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed + 1000 * i, w.q_mult))
                          for i in range(1, N_SETS)]
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    mode = args.mode
    tdt = q.dtype
    ws_bytes = cpa.cp_attention_workspace_size(w.B, w.H, w.S, w.D, w.ring_degree, w.ulysses_degree, tdt, mode)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    launches_per_step = cpa.cp_attention_launch_count(w.B, w.H, w.S, w.D, w.ring_degree, w.ulysses_degree, tdt,
                                                      mode)

    def step(i=0):
        qi, ki, vi = sets[i % N_SETS]
        cpa.cp_attention_fwd(qi, ki, vi, out, lse, w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok,
                             workspace=ws, mode=mode, stream=stream)

    step()
    torch.cuda.synchronize()
    status = cpa.cp_check_device_status()
    if status != 0:
        raise RuntimeError(f"device status after the first call: {cpa.cp_status_string(status)}")

    # parity spot check of the benchmarked output on a few rows (oracle, rank 0 only)
    parity = None
    if rank == 0:
        import oracle
        rows = np.sort(np.random.default_rng(0).choice(w.S, size=8, replace=False))
        ro, rl = oracle.attention_rows(q_h, k_h, v_h, w.scale, rows)
        go = out[:, rows].double().cpu().numpy()
        gl = lse[:, :, rows].double().cpu().numpy()
        err = max(float(np.abs(go - ro).max()), float(np.abs(gl - rl).max()))
        parity = {"rows_checked": int(len(rows)), "max_abs_err": err, "ok": bool(err <= 1e-2)}

    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[local] if os.environ.get(
        "CUDA_VISIBLE_DEVICES") else str(local)
    try:
        gpu_id = torch.cuda.get_device_properties(dev).uuid
        gpu_id = f"GPU-{gpu_id}" if not str(gpu_id).startswith("GPU-") else str(gpu_id)
    except Exception:
        pass
    clocks = clock_sampler(gpu_id)
    time.sleep(0.3)

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    # the warm-up steps run right before the timed ones, so that the timed region starts on a GPU that
    # is already busy with this work
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    # K steps back to back between one pair of events: the whole job's device time
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.time()
    clocks.mark(wall0, wall1)
    time.sleep(0.25)
    clocks.stop()
    total_ms = reduce_max(t_start.elapsed_time(t_end), world)
    ms_per_step = total_ms / args.steps
    flops_step = w.flops
    value = world * flops_step * args.steps / (total_ms * 1e-3) / 1e12
    status = cpa.cp_check_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timing: {cpa.cp_status_string(status)}")

    # e2e through host buffers: the host-buffer entry point (pinned H2D of q, k, v, the attention, D2H of
    # out and lse, with the copies of each head chunk overlapping the other chunks' attention), all timed
    q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    out_p = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_p = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (q_p, k_p, v_p))
    d2h = out_p.numel() * 4 + lse_p.numel() * 4
    host_buf = torch.empty(max(cpa.cp_attention_host_buffer_size(w.B, w.H, w.S, w.D, w.ring_degree, w.ulysses_degree,
                                                                  tdt, mode), 1), dtype=torch.uint8, device=dev)

    def e2e_step():
        cpa.cp_attention_fwd_host(q_p, k_p, v_p, out_p, lse_p, w.scale, w.ring_degree, w.ulysses_degree,
                                  w.uneven_ok, dev_buffer=host_buf, mode=mode, head_chunks=E2E_HEAD_CHUNKS,
                                  stream=stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    # back to back as well: each call copies its inputs up from host memory and its results back
    e_s.record(stream)
    for i in range(n_e2e):
        e2e_step()
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e_s.elapsed_time(e_e), world) / n_e2e
    e2e_val = world * flops_step / (e2e_ms * 1e-3) / 1e12
    step(0)  # the device call on the same inputs (the timed steps ended on another input set)
    torch.cuda.synchronize()
    if not torch.equal(out_p, out.cpu()) or not torch.equal(lse_p, lse.cpu()):
        raise RuntimeError("host-buffer call differs from the device call")

    line = None
    if rank == 0:
        peaks, peak_src = load_peaks()
        # dominant kernel: the tensor-core block-attention kernel; in the fused lap it is the
        # one launch of the step, so its average launch duration is the step's event time
        if mode == "fused" and w.dtype == "bf16":
            kernel_ms = ms_per_step
            per_launch_flops = flops_step
            scope = "attn_fwd_tc_kernel (one launch per step)"
        else:
            kernel_ms = ms_per_step
            per_launch_flops = flops_step
            scope = "whole step (several launches; merges and regroups included)"
        achieved = per_launch_flops / (kernel_ms * 1e-3) / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        traffic = profiled_traffic(w.name, mode)
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "kernel": scope,
                    "peak_source": f"{peak_src} bf16_tflops (burst: the kernel is timed alone)"}
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(w, q_h, k_h, v_h)
        sec = None
        if world == 1 and not args.no_secondary:
            sec_clocks = clock_sampler(gpu_id)
            time.sleep(0.3)
            try:
                sec = secondary(cpa, dev, flush, stream, peaks, sec_clocks)
            finally:
                time.sleep(0.25)
                sec_clocks.stop()
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": config_of(w, mode),
                "frac_of_bf16_peak": value / world / peak,
                "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms, "api": "cp_attention_fwd_host", "head_chunks": E2E_HEAD_CHUNKS},
                "gpu_launches": launches_per_step * args.steps,
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks.summary(),
                "parity_sample": parity,
                "device": {"name": torch.cuda.get_device_name(dev),
                           "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
                "secondary": sec}
    return line


def main():
    args = parse_args()
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    world, rank, local = (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                          int(os.environ.get("LOCAL_RANK", "0")))
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return 0
        line = run_reference(args, w, world, rank)
        print(json.dumps(line))
        return 0
    world, rank, local = dist_setup()
    line = run_ours(args, w, world, rank, local)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
