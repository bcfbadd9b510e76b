#!/usr/bin/env python3
"""Benchmark of gr_decode_attn on one GB300: µs per decode step and TFLOP/s
at beam width 900 over a 2048-token context (Qwen3-0.6B attention heads,
4 requests, 3 decode steps), with the roofline fraction of the dominant
kernel, an end-to-end number through host buffers, and the CPU oracle timed
on the host cores as a baseline.

One bench step = the three decode-step calls (s = 0, 1, 2) of the workload;
``value`` is the mean device time of one call (µs per decode step).  The L2
is flushed (a 2x-L2 buffer is written) before every timed call; the flush
is outside the timed interval.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]

``--op beam_select`` measures the beam-selection step instead (log_softmax +
top-W over every beam's logits, gr_beam_select): 4 requests, 900 -> 900
beams, a 151,936-token vocabulary of fp32 logits (2.19 GB per call, larger
than L2, so no flush is needed); its line carries the HBM roofline of the
per-row kernel that reads the logits.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "µs/decode-step and TFLOP/s at BW=900, Lc=2048; % of bf16/HBM roofline"
UNIT = "us/decode-step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["beam_decode_attention_gb300/csrc/gr_ctx_tc.cu", "beam_decode_attention_gb300/csrc/gr_tc_common.cuh",
                  "beam_decode_attention_gb300/csrc/gr_ptx.cuh"]
PK_KERNEL_SOURCES = ["beam_decode_attention_gb300/csrc/gr_ctx_pk.cu",
                     "beam_decode_attention_gb300/csrc/gr_tc_common.cuh",
                     "beam_decode_attention_gb300/csrc/gr_ptx.cuh"]


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=workloads.HEADLINE, choices=sorted(workloads.WORKLOAD_BY_NAME))
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip timing the other workloads (the per_config block)")
    p.add_argument("--clock-soak", type=float, default=1.5,
                   help="seconds of the same calls run under the clock sampler before the timed passes")
    p.add_argument("--op", choices=["attention", "beam_select", "trie_select", "reorder", "paged", "ragged"],
                   default="attention")
    return p.parse_args()


# ----------------------------------------------------------------------------
# algorithmic work (what the method must do, not what a kernel happens to do)


def chain_slots(inp, step):
    """Distinct (step, slot) BeamKV entries the active beams reach, per request."""
    bp, W = inp["beam_path"], inp["widths"]
    out = []
    for r in range(inp["num_requests"]):
        cur = np.arange(int(W[step]))
        n = len(cur)
        for t in range(step, 0, -1):
            cur = np.unique(bp[r, t, cur])
            n += len(cur)
        out.append(n)
    return out


def work(inp, step):
    R, Hq, Hkv, D = inp["num_requests"], inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"]
    W_s = int(inp["widths"][step])
    lens = [int(x) for x in inp["ctx_len"]]
    ctx_flops = 4.0 * W_s * Hq * D * sum(lens)
    beam_flops = 4.0 * R * W_s * Hq * D * (step + 1)
    ctx_bytes = float(sum(2 * Hkv * l * D * 2 for l in lens))
    beam_bytes = float(sum(chain_slots(inp, step)) * Hkv * 2 * D * 2)
    qo_bytes = 2.0 * R * W_s * Hq * D * 2
    lse_bytes = 4.0 * R * W_s * Hq
    path_bytes = 4.0 * R * sum(int(w) for w in inp["widths"][1:step + 1])
    return dict(flops=ctx_flops + beam_flops, ctx_flops=ctx_flops,
                bytes=ctx_bytes + beam_bytes + qo_bytes + lse_bytes + path_bytes,
                ctx_bytes=ctx_bytes)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(FALLBACK_PEAKS, source="fallback")


SELECT_KERNEL_SOURCES = ["beam_decode_attention_gb300/csrc/gr_select.cu"]


def kernel_hash(sources=None):
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, sources=None):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, only while the kernel source is unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    ent = d.get(workload)
    if not ent or ent.get("kernel_sha") != kernel_hash(sources):
        return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0], "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# CPU oracle baseline (the only place bench.py runs the oracle)


def oracle_baseline(inp, seconds):
    import oracle
    orc = oracle.Oracle()
    threads = orc.max_threads
    R = inp["num_requests"]
    total_rows = [R * int(w) for w in inp["widths"]]
    # calibrate on a few rows of the last step, then size the sample
    calib = [(r, b) for r in range(R) for b in range(0, int(inp["widths"][-1]), 97)][:max(threads, 8)]
    t0 = time.perf_counter()
    orc.decode_attn(inp, len(inp["widths"]) - 1, rows=calib)
    per_row = (time.perf_counter() - t0) / len(calib)
    est_full = per_row * sum(total_rows)
    frac = min(1.0, seconds / max(est_full, 1e-9))
    rng = np.random.default_rng(0)
    spent, rows_done, per_step_us = 0.0, 0, []
    for s, n in enumerate(total_rows):
        W_s = int(inp["widths"][s])
        k = max(1, int(round(n * frac)))
        flat = rng.choice(n, size=k, replace=False) if k < n else np.arange(n)
        rows = [(int(i // W_s), int(i % W_s)) for i in flat]
        t0 = time.perf_counter()
        orc.decode_attn(inp, s, rows=None if k == n else rows)
        dt = time.perf_counter() - t0
        spent += dt
        rows_done += k
        per_step_us.append(dt / k * n * 1e6)
    value = float(np.mean(per_step_us))
    sample = (f"{rows_done} of {sum(total_rows)} (request, beam) rows over the 3 decode steps "
              f"({100 * rows_done / sum(total_rows):.1f}%), every head; time scaled to whole steps"
              if frac < 1.0 else "every row of the 3 decode steps")
    return dict(value=value, unit=UNIT, cores=threads, kind="oracle", sample=sample,
                cpu_seconds=spent)


# ----------------------------------------------------------------------------


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    spec = workloads.WORKLOAD_BY_NAME[args.workload]
    inp = workloads.make_inputs(spec)
    per_step = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    vals, walls = [], []
    for i in range(args.warmup + args.steps):
        b = oracle_baseline(inp, per_step)
        if i >= args.warmup:
            vals.append(b["value"])
            walls.append(b["cpu_seconds"])
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # the wall time each timed step actually took (a sample of the rows);
        # `value` scales the sample to whole decode steps
        "ms_per_step": float(np.mean(walls)) * 1000.0,
        "timed_wall_s": float(np.sum(walls)),
        "extrapolated_ms_per_step": value * spec.steps / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(spec, inp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": b["cores"], "kind": "oracle",
                         "sample": b["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_of(spec, inp):
    return {"workload": spec.name, "requests": spec.num_requests, "q_heads": spec.num_q_heads,
            "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "ctx_len": [int(x) for x in inp["ctx_len"]] if spec.lc_range else spec.lc,
            "beam_widths": list(spec.widths), "decode_steps": spec.steps,
            "l2": "flushed (2x L2 buffer written) before every timed call"}


SELECT_METRIC = "µs per beam-selection call (R=4, W=900->900, V=151936, fp32 logits); % of HBM roofline"
SELECT_UNIT = "us/call"


def select_oracle_baseline(inp, next_width):
    """The selection oracle on one request, scaled to the whole call."""
    from oracle import select
    R = inp["logits"].shape[0]
    t0 = time.perf_counter()
    select.top_candidates(inp["logits"][:1], inp["beam_scores"][:1], next_width)
    dt = time.perf_counter() - t0
    return dict(value=dt * R * 1e6, unit=SELECT_UNIT, cores=1, kind="oracle",
                sample=f"request 0 of {R} (every beam and token of it), time scaled by {R}",
                cpu_seconds=dt)


def run_select_bench(args):
    import torch
    import beam_decode_attention_gb300 as gr
    cfg = workloads.SELECT_HEADLINE
    R, W, V, n = cfg["num_requests"], cfg["width"], cfg["vocab"], cfg["next_width"]
    inp = workloads.make_select_inputs(R, W, V, seed=4242)
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        vals = [select_oracle_baseline(inp, n) for _ in range(max(1, min(args.steps, 3)))]
        value = float(np.mean([v["value"] for v in vals]))
        print(json.dumps({
            "impl": "reference", "metric": SELECT_METRIC, "value": value, "unit": SELECT_UNIT, "n_gpus": 1,
            "steps": len(vals), "warmup": 0, "ms_per_step": value / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "beam_select_r4_w900_v151936", **cfg},
            "cpu_baseline": {"value": value, "unit": SELECT_UNIT, "cores": 1, "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": value, "unit": SELECT_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    torch.cuda.set_device(0)
    gr.load()
    stream = torch.cuda.current_stream()
    logits = torch.from_numpy(inp["logits"]).cuda()
    scores = torch.from_numpy(inp["beam_scores"]).cuda()
    shape = gr.SelectShape(R, W, V, n)
    ws = torch.empty(gr.gr_beam_select_workspace_size(shape), dtype=torch.uint8, device="cuda")
    par = torch.empty((R, n), dtype=torch.int32, device="cuda")
    tok = torch.empty((R, n), dtype=torch.int32, device="cuda")
    sco = torch.empty((R, n), dtype=torch.float32, device="cuda")
    for _ in range(max(3, args.warmup)):
        gr.gr_beam_select(shape, logits, scores, par, tok, sco, ws)
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    soak(torch, lambda: gr.gr_beam_select(shape, logits, scores, par, tok, sco, ws), args.clock_soak)
    call_us, rows_us = [], []
    for _ in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        gr.gr_beam_select_timed(shape, logits, scores, par, tok, sco, ws, ev)
        torch.cuda.synchronize()
        call_us.append(ev[0].elapsed_time(ev[2]) * 1000.0)
        rows_us.append(ev[0].elapsed_time(ev[1]) * 1000.0)
    clk = clocks.stop()
    if clk is not None and args.clock_soak > 0:
        clk["window"] = (f"sampled every 200 ms over a {args.clock_soak:.1f} s run of the same calls directly "
                         "before the timed calls and through them")
    value = float(np.mean(call_us))
    pk = peaks()
    logit_bytes = R * W * V * 4
    alg_bytes = logit_bytes + R * W * 4 + R * n * 12     # logits and beam scores read once, outputs
    achieved = alg_bytes / (float(np.mean(rows_us)) * 1e-6) / 1e9
    e2e = None
    if not args.no_e2e:
        h_logits = torch.from_numpy(inp["logits"]).pin_memory()
        h_scores = torch.from_numpy(inp["beam_scores"]).pin_memory()
        h_out = [torch.empty((R, n), dtype=d).pin_memory() for d in (torch.int32, torch.int32, torch.float32)]
        times = []
        for i in range(max(2, min(args.steps, 5)) + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            logits.copy_(h_logits, non_blocking=True)
            scores.copy_(h_scores, non_blocking=True)
            gr.gr_beam_select(shape, logits, scores, par, tok, sco, ws)
            for h, d in zip(h_out, (par, tok, sco)):
                h.copy_(d, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            if i > 0:
                times.append(e0.elapsed_time(e1) * 1000.0)
        e2e = {"value": float(np.mean(times)), "unit": SELECT_UNIT,
               "h2d_bytes_per_step": logit_bytes + R * W * 4, "d2h_bytes_per_step": R * n * 12,
               "note": "per call: logits and beam scores copied from pinned host memory, the three outputs back"}
    cpu = None if args.no_cpu_baseline else select_oracle_baseline(inp, n)
    line = {
        "metric": SELECT_METRIC, "value": value, "unit": SELECT_UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": value / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "beam_select_r4_w900_v151936", **cfg,
                   "l2": "inputs (2.19 GB of logits per call) larger than L2; no flush"},
        "row_kernel_us": float(np.mean(rows_us)), "merge_kernel_us": float(np.mean(call_us) - np.mean(rows_us)),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 3),
                     "traffic": recorded_traffic("beam_select_r4_w900_v151936", SELECT_KERNEL_SOURCES),
                     "kernel": "select_rows_kernel", "peak_source": pk.get("source", "measured copy")},
        "gpu_launches": 2 * args.steps, "clocks": clk, "cpu_baseline": cpu, "e2e": e2e,
    }
    print(json.dumps(line))
    return 0


TRIE_METRIC = ("µs per item-constrained selection call (R=4, W=900->900, V=151936, SID trie of 200k items, "
               "3 levels x 256 codes); % of HBM roofline")


def run_trie_bench(args):
    """Item-constrained selection (gr_trie_select): beams at trie level 1,
    so every beam has up to 256 legal tokens."""
    import torch
    import beam_decode_attention_gb300 as gr
    cfg = workloads.SELECT_TRIE_HEADLINE
    R, W, V, n = cfg["num_requests"], cfg["width"], cfg["vocab"], cfg["next_width"]
    trie = workloads.make_sid_trie(cfg["items"], cfg["levels"], cfg["codebook"], V, seed=31)
    inp = workloads.make_trie_select_inputs(R, W, V, trie, cfg["level"], seed=32)
    degs = np.diff(trie["offsets"])[inp["beam_node"]]
    legal = int(degs.sum())
    conf = {"workload": "trie_select_r4_w900_v151936_sid3x256", **cfg,
            "legal_candidates": legal, "l2": "logits 2.19 GB, of which only the legal entries are read; no flush"}
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        from oracle import select
        t0 = time.perf_counter()
        select.trie_select(inp["logits"][:1], inp["beam_scores"][:1], inp["beam_node"][:1], trie["offsets"],
                           trie["tokens"], trie["children"], n)
        value = (time.perf_counter() - t0) * R * 1e6
        print(json.dumps({
            "impl": "reference", "metric": TRIE_METRIC, "value": value, "unit": SELECT_UNIT, "n_gpus": 1,
            "steps": 1, "warmup": 0, "ms_per_step": value / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": conf,
            "cpu_baseline": {"value": value, "unit": SELECT_UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"request 0 of {R}, time scaled by {R}"},
            "e2e": {"value": value, "unit": SELECT_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    torch.cuda.set_device(0)
    gr.load()
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    logits, scores, bn = d(inp["logits"]), d(inp["beam_scores"]), d(inp["beam_node"])
    off, tok, ch = d(trie["offsets"]), d(trie["tokens"]), d(trie["children"])
    shape = gr.TrieSelectShape(R, W, V, n, trie["num_nodes"], len(trie["tokens"]))
    ws = torch.empty(gr.gr_trie_select_workspace_size(shape), dtype=torch.uint8, device="cuda")
    par = torch.empty((R, n), dtype=torch.int32, device="cuda")
    tk, nd = torch.empty_like(par), torch.empty_like(par)
    sc = torch.empty((R, n), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(max(3, args.warmup)):
        gr.gr_trie_select(shape, logits, scores, bn, off, tok, ch, par, tk, sc, nd, ws)
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()

    def one():
        flush.zero_()
        gr.gr_trie_select(shape, logits, scores, bn, off, tok, ch, par, tk, sc, nd, ws)

    soak(torch, one, args.clock_soak)
    times = []
    for _ in range(args.steps):
        flush.zero_()   # the legal logits are a few MB: flush L2 before each call
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gr.gr_trie_select(shape, logits, scores, bn, off, tok, ch, par, tk, sc, nd, ws)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0)
    clk = clocks.stop()
    if clk is not None and args.clock_soak > 0:
        clk["window"] = (f"sampled every 200 ms over a {args.clock_soak:.1f} s run of the same calls directly "
                         "before the timed calls and through them")
    value = float(np.mean(times))
    pk = peaks()
    # algorithmic bytes: the legal logits, their edge tokens and children, the
    # beams' nodes, scores and trie offsets, and the outputs
    alg = legal * 4 * 3 + R * W * 12 + R * n * 16
    conf["l2"] = "flushed (256 MB buffer written) before every timed call"
    line = {
        "metric": TRIE_METRIC, "value": value, "unit": SELECT_UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": value / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": conf,
        "roofline": {"bound": "hbm", "achieved": round(alg / (value * 1e-6) / 1e9, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(alg / (value * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                     "traffic": recorded_traffic(conf["workload"], SELECT_KERNEL_SOURCES),
                     "kernel": "whole call (trie_rows_warp_kernel, trie_rows_kernel, select_merge_kernel)",
                     "peak_source": pk.get("source", "measured copy")},
        "gpu_launches": 3 * args.steps, "clocks": clk, "cpu_baseline": None, "e2e": None,
    }
    print(json.dumps(line))
    return 0


def run_reorder_bench(args):
    """BeamPath indirection against the reordered per-beam cache (xGR's
    alternative) on the headline workload: per decode step, the attention
    call through BeamPath, against gr_beam_reorder (out of place) or
    gr_beam_reorder_inplace plus the attention call on the reordered cache
    with the identity path; and the BeamKV append of the step's K/V.  L2
    flushed before each call."""
    import torch
    import beam_decode_attention_gb300 as gr
    spec = workloads.WORKLOAD_BY_NAME[workloads.HEADLINE]
    inp = workloads.make_inputs(spec)
    torch.cuda.set_device(0)
    gr.load()
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()
    shape = gr.Shape.of(inp)
    widths = [int(w) for w in inp["widths"]]
    ck, cv, cl = up(inp["ctx_k"]), up(inp["ctx_v"]), up(inp["ctx_len"])
    bk, bv, bp = up(inp["beam_k"]), up(inp["beam_v"]), up(inp["beam_path"])
    ok, ov, op = torch.empty_like(bk), torch.empty_like(bv), torch.empty_like(bp)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res = {}
    for step in range(len(widths)):
        q = up(inp["q"][step])
        R, W_s, Hq, D = spec.num_requests, widths[step], spec.num_q_heads, spec.head_dim
        out = torch.empty(R * W_s * Hq * D, dtype=torch.int16, device="cuda")
        lse = torch.empty(R * W_s * Hq, dtype=torch.float32, device="cuda")
        flat = [W_s] * len(widths)
        ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(shape, widths, step)), dtype=torch.uint8,
                         device="cuda")
        t_path, t_reorder, t_flat, t_inplace, t_append = [], [], [], [], []
        kn = torch.randn(R * W_s * spec.num_kv_heads * D, device="cuda").to(torch.bfloat16).view(torch.int16)
        vn = torch.randn(R * W_s * spec.num_kv_heads * D, device="cuda").to(torch.bfloat16).view(torch.int16)
        for i in range(max(3, args.warmup) + args.steps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            gr.gr_decode_attn(shape, q, ck, cv, cl, bk, bv, bp, widths, step, out, lse, ws)
            e[1].record()
            flush.zero_()
            f = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            f[0].record()
            gr.gr_beam_reorder(shape, bk, bv, bp, widths, step, ok, ov, op)
            f[1].record()
            gr.gr_decode_attn(shape, q, ck, cv, cl, ok, ov, op, flat, step, out, lse, ws)
            f[2].record()
            # the in-place reorder on a fresh copy of the cache (a second
            # call would find the identity path and move nothing)
            ik, iv, ip = bk.clone(), bv.clone(), bp.clone()
            flush.zero_()
            h = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            h[0].record()
            gr.gr_beam_reorder_inplace(shape, ik, iv, ip, widths, step)
            h[1].record()
            flush.zero_()
            a = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            a[0].record()
            gr.gr_beam_append(shape, widths, step, kn, vn, ik, iv)
            a[1].record()
            torch.cuda.synchronize()
            del ik, iv, ip
            if i >= max(3, args.warmup):
                t_path.append(e[0].elapsed_time(e[1]) * 1000)
                t_reorder.append(f[0].elapsed_time(f[1]) * 1000)
                t_flat.append(f[1].elapsed_time(f[2]) * 1000)
                t_inplace.append(h[0].elapsed_time(h[1]) * 1000)
                t_append.append(a[0].elapsed_time(a[1]) * 1000)
        row_bytes = spec.num_kv_heads * D * 2
        # in place: K and V of every level below `step`, each source row read
        # once and each beam's row written once
        inplace_bytes = 2 * R * sum(widths[t] + W_s for t in range(step)) * row_bytes
        append_bytes = 2 * 2 * R * W_s * row_bytes
        res[step] = (float(np.mean(t_path)), float(np.mean(t_reorder)), float(np.mean(t_flat)),
                     float(np.mean(t_inplace)), float(np.mean(t_append)), inplace_bytes, append_bytes)
    line = {
        "metric": "µs per decode step: attention through BeamPath vs reorder + attention on the reordered cache",
        "value": float(np.mean([v[0] for v in res.values()])), "unit": "us/decode-step", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "higher_is_better": False, "dtype": "bf16",
        "data": "synthetic", "config": config_of(spec, inp),
        "per_step": {str(k): {"beampath_us": round(v[0], 2), "reorder_us": round(v[1], 2),
                              "attention_on_reordered_us": round(v[2], 2),
                              "reorder_total_us": round(v[1] + v[2], 2),
                              "reorder_inplace_us": round(v[3], 2),
                              "reorder_inplace_gbs": round(v[5] / v[3] / 1e3, 1) if v[3] > 0 else None,
                              "inplace_total_us": round(v[3] + v[2], 2),
                              "append_us": round(v[4], 2),
                              "append_gbs": round(v[6] / v[4] / 1e3, 1)} for k, v in res.items()},
        "hbm_peak_gbs": peaks().get("hbm_gbs"),
    }
    print(json.dumps(line))
    return 0


RAGGED_WIDTHS = (900, 600, 300, 128)   # the four headline requests' widths in the ragged layout bench


def run_layout_bench(args):
    """The context and width layouts on the headline geometry, each against
    the dense call on the same data, L2 flushed before every call:
      paged   ContextKV in 128-key pages of a shuffled pool through a block table;
      ragged  per-request widths 900 / 600 / 300 / 128 in one batch, against the
              dense call over the same tensors at the largest width.
    TFLOP/s count the rows each call computes (the ragged call: the active rows)."""
    import torch
    import beam_decode_attention_gb300 as gr
    spec = workloads.WORKLOAD_BY_NAME[workloads.HEADLINE]
    torch.cuda.set_device(0)
    gr.load()
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()
    if args.op == "ragged":
        inp, W = workloads.make_ragged(spec, [[w] * spec.steps for w in RAGGED_WIDTHS])
    else:
        inp, W = workloads.make_inputs(spec), None
    shape = gr.Shape.of(inp)
    widths = [int(w) for w in inp["widths"]]
    ck, cv, cl = up(inp["ctx_k"]), up(inp["ctx_v"]), up(inp["ctx_len"])
    bk, bv, bp = up(inp["beam_k"]), up(inp["beam_v"]), up(inp["beam_path"])
    if args.op == "paged":
        kp, table, ppr, P = workloads.paged_pool(inp["ctx_k"], 128, 8, seed=1)
        vp, _, _, _ = workloads.paged_pool(inp["ctx_v"], 128, 8, seed=1)
        pages = gr.CtxPages(128, P, ppr)
        kp_d, vp_d, tb_d = up(kp), up(vp), up(table)
    else:
        wdev = np.zeros((spec.num_requests, spec.steps), np.int32)
        wdev[:, :] = W
        wdev_d = up(wdev)
    flush = torch.empty(2 * torch.cuda.get_device_properties(0).L2_cache_size, dtype=torch.uint8, device="cuda")
    R, Hq, D = spec.num_requests, spec.num_q_heads, spec.head_dim
    lc = [int(x) for x in inp["ctx_len"]]
    res = {}
    for step in range(spec.steps):
        q = up(inp["q"][step])
        W_s = widths[step]
        out = torch.empty(R * W_s * Hq * D, dtype=torch.int16, device="cuda")
        lse = torch.empty(R * W_s * Hq, dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(shape, widths, step)), dtype=torch.uint8,
                         device="cuda")

        def dense():
            gr.gr_decode_attn(shape, q, ck, cv, cl, bk, bv, bp, widths, step, out, lse, ws)

        def layout():
            if args.op == "paged":
                gr.gr_decode_attn_paged(shape, pages, q, kp_d, vp_d, cl, tb_d, bk, bv, bp, widths, step, out, lse, ws)
            else:
                gr.gr_decode_attn_ragged(shape, q, ck, cv, cl, bk, bv, bp, W.tolist(), wdev_d, step, out, lse, ws)

        t_dense, t_layout = [], []
        for i in range(max(3, args.warmup) + args.steps):
            for fn, acc in ((dense, t_dense), (layout, t_layout)):
                flush.zero_()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record()
                fn()
                e[1].record()
                torch.cuda.synchronize()
                if i >= max(3, args.warmup):
                    acc.append(e[0].elapsed_time(e[1]) * 1000)
        rows = [W_s] * R if W is None else [int(W[r, step]) for r in range(R)]
        flops = sum(4.0 * D * Hq * rows[r] * (lc[r] + step + 1) for r in range(R))
        dense_flops = sum(4.0 * D * Hq * W_s * (lc[r] + step + 1) for r in range(R))
        res[step] = (float(np.mean(t_layout)), float(np.mean(t_dense)), flops, dense_flops)
    err = gr.gr_get_device_error()
    value = float(np.mean([v[0] for v in res.values()]))
    line = {
        "metric": ("µs per decode step, " + ("paged ContextKV (128-key pages, shuffled pool)" if args.op == "paged"
                                            else "per-request widths 900/600/300/128 in one batch")
                   + " against the dense call"),
        "value": round(value, 3), "unit": "us/decode-step", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(spec, inp), layout=args.op,
                       **({"request_widths": list(RAGGED_WIDTHS)} if args.op == "ragged" else {"page_size": 128})),
        "per_step": {str(k): {"layout_us": round(v[0], 2), "dense_us": round(v[1], 2),
                              "layout_tflops": round(v[2] / v[0] * 1e-6, 1),
                              "dense_tflops": round(v[3] / v[1] * 1e-6, 1)} for k, v in res.items()},
        "dense_value": round(float(np.mean([v[1] for v in res.values()])), 3),
        "device_error": err,
    }
    print(json.dumps(line))
    return 0 if err == 0 else 1


def soak(torch, fn, seconds):
    """Runs fn() back to back for about `seconds`, so that a clock sampler
    started before sees the load the timed calls that follow run under."""
    if seconds <= 0:
        return
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(8):
            fn()
        torch.cuda.synchronize()


def attention_run(gr, torch, spec, steps, warmup, soak_s=0.0, clocks=None):
    """Times the decode-step calls of one workload: `warmup` untimed passes,
    then exactly `steps` timed passes over its decode steps, each call
    bracketed by CUDA events on the launching stream (the context kernel
    separately), with the L2 flushed (a 2x-L2 buffer written) before every
    call.  With soak_s > 0 the same calls run for that long before the timed
    passes while `clocks` samples (so the sampler sees the load; the timed
    passes follow inside the same sampling window)."""
    inp = workloads.make_inputs(spec)
    S = spec.steps
    dev = torch.device("cuda:0")

    def up(a):
        a = a.view(np.int16) if a.dtype == np.uint16 else a
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    shape = gr.Shape.of(inp)
    widths = [int(w) for w in inp["widths"]]
    ctx_k, ctx_v, ctx_len = up(inp["ctx_k"]), up(inp["ctx_v"]), up(inp["ctx_len"])
    beam_k, beam_v, beam_path = up(inp["beam_k"]), up(inp["beam_v"]), up(inp["beam_path"])
    qs = [up(x) for x in inp["q"]]
    R, Hq, D = spec.num_requests, spec.num_q_heads, spec.head_dim
    outs = [torch.empty(R * widths[s] * Hq * D, dtype=torch.int16, device=dev) for s in range(S)]
    lses = [torch.empty(R * widths[s] * Hq, dtype=torch.float32, device=dev) for s in range(S)]
    ws_bytes = max(gr.gr_decode_attn_workspace_size(shape, widths, s) for s in range(S))
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    plans = [gr.gr_decode_attn_plan(shape, widths, s) for s in range(S)]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    works = [work(inp, s) for s in range(S)]

    def call(s, ev=None):
        if ev is None:
            gr.gr_decode_attn(shape, qs[s], ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, s,
                              outs[s], lses[s], ws, stream=stream)
        else:
            gr.gr_decode_attn_timed(shape, qs[s], ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path,
                                    widths, s, outs[s], lses[s], ws, ev, stream=stream)

    for _ in range(warmup):
        for s in range(S):
            flush.zero_()
            call(s)
    torch.cuda.synchronize()
    if gr.gr_get_device_error() != 0:
        raise RuntimeError(f"device error during the warm-up of {spec.name}")

    # events[k][s] = [before the call, after the context kernel, after the
    # call]; the middle one only when a second kernel follows (each event
    # record adds about 2 us of device time between its neighbours, so a
    # one-kernel call is bracketed by two events and its kernel time is the
    # call time)
    one_kernel = [p["kernels"] == 1 for p in plans]
    events = [[[torch.cuda.Event(enable_timing=True), None if one_kernel[s] else torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)] for s in range(S)] for _ in range(steps)]
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    if soak_s > 0:
        t_end = time.perf_counter() + soak_s
        while time.perf_counter() < t_end:
            for s in range(S):
                flush.zero_()
                call(s)
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    for k in range(steps):
        for s in range(S):
            flush.zero_()
            call(s, events[k][s])
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks is not None else None
    if gr.gr_get_device_error() != 0:
        raise RuntimeError(f"device error during the timed passes of {spec.name}")

    call_us = np.array([[1000.0 * events[k][s][0].elapsed_time(events[k][s][2]) for s in range(S)]
                        for k in range(steps)])
    ctx_us = np.array([[1000.0 * events[k][s][0].elapsed_time(events[k][s][2 if one_kernel[s] else 1])
                        for s in range(S)] for k in range(steps)])
    per_step_us = call_us.mean(axis=0)
    per_step_ctx_us = ctx_us.mean(axis=0)
    pk = peaks()
    total_flops = sum(w["flops"] for w in works)
    ctx_flops = sum(w["ctx_flops"] for w in works)
    achieved_tf = ctx_flops / (per_step_ctx_us.sum() * 1e-6) / 1e12
    roof_us = [max(w["flops"] / (pk["bf16_tflops"] * 1e12), w["bytes"] / (pk["hbm_gbs"] * 1e9)) * 1e6
               for w in works]
    bound = ["tensor" if w["flops"] / (pk["bf16_tflops"] * 1e12) >= w["bytes"] / (pk["hbm_gbs"] * 1e9)
             else "hbm" for w in works]
    # the context kernel against its own bound: its FLOPs at the bf16 peak, or
    # its bytes at HBM bandwidth when that is slower (it reads everything the
    # call reads: the per-beam stage and the merge are fused into it)
    ctx_roof_us = [max(w["ctx_flops"] / (pk["bf16_tflops"] * 1e12), w["bytes"] / (pk["hbm_gbs"] * 1e9)) * 1e6
                   for w in works]
    return dict(
        inp=inp, shape=shape, widths=widths, ws=ws, stream=stream, plans=plans, clocks=clk, works=works,
        value=float(per_step_us.mean()),
        per_step_us=[round(float(x), 2) for x in per_step_us],
        per_step_median_us=[round(float(x), 2) for x in np.median(call_us, axis=0)],
        per_step_min_us=[round(float(x), 2) for x in call_us.min(axis=0)],
        per_step_ctx_us=[round(float(x), 2) for x in per_step_ctx_us],
        tflops=round(total_flops / (per_step_us.sum() * 1e-6) / 1e12, 2),
        ctx_tflops=round(achieved_tf, 2),
        ctx_gbs=round(sum(w["bytes"] for w in works) / (per_step_ctx_us.sum() * 1e-6) / 1e9, 1),
        roofline_us=[round(x, 2) for x in roof_us], bound=bound,
        call_frac_per_step=[round(a / b, 4) for a, b in zip(roof_us, per_step_us)],
        call_frac=round(sum(roof_us) / float(per_step_us.sum()), 4),
        ctx_frac=round(sum(ctx_roof_us) / float(per_step_ctx_us.sum()), 4),
        ctx_frac_of_bf16=round(achieved_tf / pk["bf16_tflops"], 4),
        launches=sum(p["kernels"] for p in plans) * steps,
    )


def main():
    args = parse_args()
    if args.gpus != 1:
        print(json.dumps({"error": "every call runs on one GPU (independent requests: replicas only); --gpus must be 1"}))
        return 2
    if args.op == "beam_select":
        return run_select_bench(args)
    if args.op == "trie_select":
        return run_trie_bench(args)
    if args.op == "reorder":
        return run_reorder_bench(args)
    if args.op in ("paged", "ragged"):
        return run_layout_bench(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import beam_decode_attention_gb300 as gr

    torch.cuda.set_device(0)
    spec = workloads.WORKLOAD_BY_NAME[args.workload]
    pk = peaks()
    clocks = ClockSampler()
    res = attention_run(gr, torch, spec, args.steps, args.warmup, soak_s=args.clock_soak, clocks=clocks)
    # the dominant kernel is the one of the slowest decode step
    slowest = int(np.argmax(res["per_step_us"]))
    persistent = bool(res["plans"][slowest].get("persistent"))
    kname = ("ctx_pk_kernel (persistent; context stage, fused per-beam stage and merge)" if persistent else
             "ctx_tc_kernel (context stage, fused per-beam stage and merge)")
    traffic = recorded_traffic(spec.name, PK_KERNEL_SOURCES if persistent else None)
    if res["bound"][slowest] == "hbm":
        roofline = {"bound": "hbm", "achieved": res["ctx_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(res["ctx_gbs"] / pk["hbm_gbs"], 4), "traffic": traffic, "kernel": kname,
                    "peak_source": f"{pk['source']} HBM copy"}
    else:
        roofline = {"bound": "tensor", "achieved": res["ctx_tflops"], "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": res["ctx_frac_of_bf16"], "traffic": traffic, "kernel": kname,
                    "peak_source": f"{pk['source']} bf16 burst"}
    call_roofline = {"roofline_us_per_step": res["roofline_us"], "measured_us_per_step": res["per_step_us"],
                     "bound_per_step": res["bound"], "frac_per_step": res["call_frac_per_step"],
                     "frac": res["call_frac"]}

    per_config = {}
    if not args.no_per_config:
        for other in workloads.WORKLOADS[1:]:
            if other.name == spec.name:
                continue
            o = attention_run(gr, torch, other, max(3, min(args.steps, 10)), 3)
            # the kernel of the slowest decode step dominates the call
            slowest = int(np.argmax(o["per_step_us"]))
            persistent = bool(o["plans"][slowest].get("persistent"))
            per_config[other.name] = {
                "dominant_kernel": "ctx_pk_kernel" if persistent else "ctx_tc_kernel",
                "traffic": recorded_traffic(other.name, PK_KERNEL_SOURCES if persistent else None),
                "us_per_decode_step": o["per_step_us"], "median_us": o["per_step_median_us"],
                "min_us": o["per_step_min_us"], "mean_us": round(o["value"], 3), "tflops": o["tflops"],
                "roofline_us_per_step": o["roofline_us"], "bound_per_step": o["bound"],
                "call_roofline_frac": o["call_frac"], "context_kernel_us": o["per_step_ctx_us"],
                "context_kernel_frac": o["ctx_frac"], "context_kernel_frac_of_bf16": o["ctx_frac_of_bf16"],
                "plan": [{k: p[k] for k in ("n_splits", "context_ctas", "kernels")} for p in o["plans"]],
                "timed_passes": max(3, min(args.steps, 10)),
            }
            del o

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(gr, torch, res["inp"], res["shape"], res["widths"], res["ws"], res["stream"], args)

    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_baseline(res["inp"], args.cpu_seconds)

    clk = res["clocks"]
    if clk is not None:
        clk["window"] = (f"sampled every 200 ms over a {args.clock_soak:.1f} s run of the same calls directly "
                         "before the timed passes and through them")
    line = {
        "metric": METRIC, "value": round(res["value"], 3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sum(res["per_step_us"]) / 1000.0, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(spec, res["inp"]),
        "tflops": res["tflops"], "us_per_decode_step": res["per_step_us"],
        "us_per_decode_step_median": res["per_step_median_us"], "us_per_decode_step_min": res["per_step_min_us"],
        "context_kernel_us": res["per_step_ctx_us"],
        "roofline": roofline, "call_roofline": call_roofline, "per_config": per_config,
        "plan": res["plans"], "gpu_launches": res["launches"], "clocks": clk,
        "cpu_baseline": cpu, "e2e": e2e,
    }
    print(json.dumps(line))
    return 0


def end_to_end(gr, torch, inp, shape, widths, ws, stream, args):
    """The same calls from pinned host buffers: each call's inputs are copied
    host->device, the call runs, out and lse come back device->host."""
    S = len(widths)
    R, Hq, D = inp["num_requests"], inp["num_q_heads"], inp["head_dim"]

    def pin(a):
        a = a.view(np.int16) if a.dtype == np.uint16 else a
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    host = {k: pin(inp[k]) for k in ("ctx_k", "ctx_v", "ctx_len", "beam_k", "beam_v", "beam_path")}
    host_q = [pin(x) for x in inp["q"]]
    devb = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    dev_q = [torch.empty_like(x, device="cuda") for x in host_q]
    outs = [torch.empty(R * widths[s] * Hq * D, dtype=torch.int16, device="cuda") for s in range(S)]
    lses = [torch.empty(R * widths[s] * Hq, dtype=torch.float32, device="cuda") for s in range(S)]
    host_out = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
    host_lse = [torch.empty_like(x, device="cpu").pin_memory() for x in lses]
    h2d = [sum(v.numel() * v.element_size() for v in host.values()) + host_q[s].numel() * 2
           for s in range(S)]
    d2h = [outs[s].numel() * 2 + lses[s].numel() * 4 for s in range(S)]

    def one(s):
        for k in host:
            devb[k].copy_(host[k], non_blocking=True)
        dev_q[s].copy_(host_q[s], non_blocking=True)
        gr.gr_decode_attn(shape, dev_q[s], devb["ctx_k"], devb["ctx_v"], devb["ctx_len"],
                          devb["beam_k"], devb["beam_v"], devb["beam_path"], widths, s, outs[s],
                          lses[s], ws, stream=stream)
        host_out[s].copy_(outs[s], non_blocking=True)
        host_lse[s].copy_(lses[s], non_blocking=True)

    for _ in range(args.warmup):
        for s in range(S):
            one(s)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        for s in range(S):
            one(s)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (steps * S)
    return {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": int(np.mean(h2d)),
            "d2h_bytes_per_step": int(np.mean(d2h)),
            "note": "per decode-step call: every input the call reads copied from pinned host memory"}


if __name__ == "__main__":
    sys.exit(main())
