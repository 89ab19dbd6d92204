#!/usr/bin/env python
"""Benchmark of the unified paged-KV attention forward on GB300.

One step = one ua_forward over the whole batch of the chosen workload (every
kernel of the path: prefill, split-KV decode, combine). Default workload: the
pure-decode batch (64 sequences, kv_len ~ U[512, 4096], 32 query / 8 KV heads,
head_dim 128, bf16, block_size 16); metric: KV-read GB/s (algorithmic bytes:
every visible K/V row once, plus Q, output, page tables and lengths).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
                    [--impl ours|reference]

Under torchrun each rank runs its own independent batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line. `--impl reference`
times the fp64 CPU oracle (the only other implementation of this path) on a
bounded sample of the same workload, on the host cores.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
WORKLOAD_NAMES = {
    1: "tiny mixed batch: 3 seqs, q [1,5,17], kv [40,130,300], 4/4 heads, d64, bf16, bs16",
    2: "pure decode: 64 seqs, q 1, kv U[512,4096], 32/8 heads, d128, bf16, bs16",
    3: "mixed: 8 prefill (q U[512,2048], ctx U[0,1024]) + 120 decode (kv U[1024,8192]), "
       "32/8 heads, d128, bf16, bs16",
    4: "dense causal prefill: 4 seqs x 4096, 32/32 heads, d128, bf16, bs128, identity table",
    5: "long decode fp8: 8 seqs, kv 131072, 64/8 heads, d128, fp8 e4m3 KV, bs16",
    6: "dense causal prefill over an fp8 cache: 4 seqs x 4096, 32/32 heads, d128, fp8 e4m3 KV, "
       "bs16, random table (not a benchmark configuration: measures the fp8 prefill path)",
    7: "uniform decode: 32 seqs, q 1, kv 8192, 32/8 heads, d128, bf16, bs16 (not a benchmark "
       "configuration: measures split sizing on equal lengths)",
    8: "pure decode at head_dim 256: 64 seqs, q 1, kv U[512,4096], 32/8 heads, bf16, bs16 "
       "(not a benchmark configuration: measures the head_dim 256 decode path)",
    9: "dense causal prefill at head_dim 256: 4 seqs x 4096, 32/32 heads, bf16, bs128, identity "
       "table (not a benchmark configuration: measures the head_dim 256 prefill kernel)",
    10: "pure decode at head_dim 96: 64 seqs, q 1, kv U[512,4096], 32/8 heads, bf16, bs16 "
        "(not a benchmark configuration: measures the decode kernel at a non-power-of-two "
        "head dim)",
    11: "dense causal prefill at head_dim 192: 4 seqs x 4096, 32/32 heads, bf16, bs128, "
        "identity table (not a benchmark configuration: measures the head_dim 192 prefill)",
}
FLOP_CONFIGS = (4, 6, 9, 11)   # prefill-bound workloads, reported in TFLOP/s


def _seq_work(case):
    """Per sequence: (bytes, flops) of one forward without the length arrays --
    every visible K/V row once per KV head, Q and the output once, the used
    page-table entries; flops = 4 * d per (query head, visible key)."""
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    d, hq, hkv = case.head_dim, case.num_q_heads, case.num_kv_heads
    out = []
    for s in range(case.num_seqs):
        ql, kv = cu[s + 1] - cu[s], kvl[s]
        if ql == 0:
            out.append((0, 0))
            continue
        ctx = kv - ql
        lo = max(0, ctx - case.window + 1) if case.window > 0 else 0
        vis_pairs = 0
        for i in range(ql):
            pos = ctx + i
            hi = pos + 1 if case.causal else kv
            l0 = max(0, pos - case.window + 1) if case.window > 0 else 0
            vis_pairs += hi - l0
        byts = (kv - lo) * hkv * d * elt * 2 + 2 * ql * hq * d * 2 + -(-kv // case.block_size) * 4
        out.append((byts, 4 * d * hq * vis_pairs))
    return out


def algorithmic_work(case):
    """(bytes, flops) one forward must move / compute: the per-sequence work
    of _seq_work plus the two length arrays."""
    per = _seq_work(case)
    return (sum(b for b, _ in per) + (2 * case.num_seqs + 1) * 4, sum(f for _, f in per))


def units_work(case, units, per=None):
    """(bytes, flops) of (sequence, KV head) oracle units: each KV head of a
    sequence carries 1 / Hkv of that sequence's work."""
    per = per if per is not None else _seq_work(case)
    h = case.num_kv_heads
    return (sum(per[s][0] for s, _ in units) / h, sum(per[s][1] for s, _ in units) / h)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (read only) while the block runs; summary() keeps
    the samples inside the window given by mark_load() / end_load()."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_load(self):
        self.window = [time.time(), None]

    def end_load(self):
        if self.window:
            self.window[1] = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        import datetime
        sm, mx, power, reasons, all_n = [], None, [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            all_n += 1
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if self.window and ts is not None and not (
                    self.window[0] - 0.05 <= ts <= (self.window[1] or ts) + 0.05):
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_total": all_n,
                "power_w_max": max(power) if power else None,
                "window_s": (self.window[1] - self.window[0])
                if self.window and self.window[1] else None}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline; never on the GPU path)
# ---------------------------------------------------------------------------

def _oracle_units(case, seed=0):
    """Every (sequence, KV head) unit of the workload in a seeded random order,
    so that a time-bounded sample mixes long and short sequences as the
    workload does."""
    import random
    from oracle import pool
    units = pool.units_of(case.cu_query_lens.tolist(), case.num_kv_heads)
    random.Random(seed).shuffle(units)
    return units


def oracle_throughput(cfg, case, budget_s=10.0, rounds=1, workers=None):
    """Time the fp64 oracle on every host core (oracle.pool: one process per
    core, one thread each) on (sequence, KV head) units of the workload for
    about budget_s of wall time per round. Returns ([rate per round], cores,
    sample description, [(bytes, flops, seconds)] per round)."""
    from oracle import pool
    per = _seq_work(case)
    per_round, n = pool.time_units(case.raw(), case.block_size, case.scale, budget_s,
                                   kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                   v_scale=case.v_scale, causal=case.causal,
                                   window=case.window, workers=workers,
                                   units=_oracle_units(case), rounds=rounds)
    rates, raw = [], []
    for done, wall in per_round:
        b, f = units_work(case, done, per)
        rates.append(_rate(cfg, b, f, wall))
        raw.append((b, f, wall))
    total_units = case.num_seqs * case.num_kv_heads
    done0 = per_round[0][0]
    sample = (f"{len(done0)} (sequence, KV head) units of the same workload "
              f"({len(set(done0))} distinct of {total_units}, seeded random order) in "
              f"{per_round[0][1]:.1f} s of wall time on {n} worker processes, one thread each")
    return rates, n, sample, raw


def _metric_for(cfg):
    if cfg in FLOP_CONFIGS:
        return "prefill TFLOP/s (algorithmic causal flops / step time)", "TFLOP/s"
    return "decode KV-read GB/s (algorithmic K/V+Q+O bytes / step time)", "GB/s"


def _dtype_for(case):
    return "fp8e4m3 KV -> f16 MMA, fp32 accumulate" if case.kv_dtype == "fp8_e4m3" else \
        "bf16 MMA, fp32 accumulate"


def _rate(cfg, byts, flops, seconds):
    return (flops / seconds / 1e12) if cfg in FLOP_CONFIGS else (byts / seconds / 1e9)


# ---- replicas across ranks (weak scaling: an independent batch per GPU) ----

def _with_window(case, window):
    """The workload with a left sliding window of `window` keys (0: none)."""
    return dataclasses.replace(case, window=int(window)) if window else case


def rank_case(cfg, rank):
    """This rank's batch: the workload drawn with seed = rank."""
    import workloads as W
    return W.CONFIGS[cfg](seed=rank)


def max_over_ranks(value, world, device="cpu"):
    """Largest value over the ranks (the job's step time is its slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, world, device="cpu"):
    """Sum over the ranks (work units the whole job processed)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def run_reference(args):
    """The oracle as the reference arm: host cores only, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import workloads as W
    cfg = args.workload
    case = _with_window(W.CONFIGS[cfg](), getattr(args, "window", 0))
    metric, unit = _metric_for(cfg)
    step_budget = max(0.5, min(2.0, 60.0 / max(1, args.steps + args.warmup)))
    if getattr(args, "op", "attention") == "append":
        return _reference_append(args, case, step_budget)
    _, cores, _, raw = oracle_throughput(cfg, case, budget_s=step_budget,
                                         rounds=args.warmup + args.steps)
    timed = raw[args.warmup:]
    tot_b = sum(r[0] for r in timed)
    tot_f = sum(r[1] for r in timed)
    tot_t = sum(r[2] for r in timed)
    value = _rate(cfg, tot_b, tot_f, tot_t)
    sample = (f"each step: (sequence, KV head) units of the workload in a seeded random order "
              f"for about {step_budget:.1f} s of wall time on {cores} worker processes "
              f"(one thread each)")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, len(timed)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": WORKLOAD_NAMES[cfg],
                   "parallelism": f"host, {cores} processes x 1 thread",
                   **({"window": case.window} if case.window else {})},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _traffic_record(kernel: str, cfg):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources (profiles/traffic.json: {key: {"source_hash", "bytes"}}).
    Returns (bytes or None, note, {"current": digest, "record": digest})."""
    from paged_kv_attention_unified_gb300 import build as B
    cur = B.kernel_digest(kernel)
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}/workload{cfg}")
    except Exception:
        rec = None
    digests = {"current": cur, "record": rec.get("source_hash") if rec else None}
    if rec and rec.get("source_hash") == cur:
        return float(rec["bytes_per_launch"]), rec.get("note"), digests
    return None, None, digests


def _timed_steps(n, step, stream, flush):
    """Device milliseconds of n back-to-back steps: one event pair around all
    of them, or one per step when the L2 is flushed between steps."""
    import torch
    if flush is None:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)
    ms = 0.0
    for _ in range(n):
        flush.zero_()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        step()
        t1.record(stream)
        torch.cuda.synchronize()
        ms += t0.elapsed_time(t1)
    return ms


def measure_attention(cfg, args, rank, world, with_cpu, soak_s, cpu_budget):
    """One workload through ua_forward: W warm-up steps, a soak of at least
    soak_s (the same step back to back; gives the sustained rate and the clock
    record under load), then exactly K timed steps with per-kernel events, the
    roofline of the dominant kernel, end to end through the C ABI with host
    buffers, and the oracle on the host cores. Returns the result fields."""
    import torch
    import paged_kv_attention_unified_gb300 as ua
    from paged_kv_attention_unified_gb300 import torch_utils as tu

    case = _with_window(rank_case(cfg, rank), args.window)   # weak scaling: one batch per GPU
    per = _seq_work(case)
    byts, flops = algorithmic_work(case)
    hbm_peak, tf_peak, peak_src = _peaks()
    cpu = None
    if with_cpu:
        rates, cores, sample, _ = oracle_throughput(cfg, case, budget_s=cpu_budget)
        cpu = {"value": rates[0], "unit": _metric_for(cfg)[1], "cores": cores, "kind": "oracle",
               "sample": sample}

    b = tu.to_device(case)
    plan = tu.make_plan(b, num_splits=args.num_splits)
    plan.set_unified_max(args.unified_max)
    if args.prefill_ctas:
        ua.ua_plan_set_prefill_ctas(plan.handle, args.prefill_ctas)
    f8p = bool(getattr(args, "fp8_products", False)) and case.kv_dtype == "fp8_e4m3"
    if f8p:
        ua.ua_plan_set_fp8_products(plan.handle, True)
        # e4m3 operands: the fp8 dense peak, the measured bf16 one times the
        # nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
        tf_peak *= 2.0
    info = plan.info
    out = b.new_out()
    stream = torch.cuda.current_stream()
    step = lambda: tu.forward(plan, b, out)
    ua.ua_plan_set_profiling(plan.handle, False)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flush = None
    if byts < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.mark_load()
        # soak: chunks of about 0.1 s until soak_s has run
        per_step_ms = max(1e-3, _timed_steps(1, step, stream, flush))
        chunk = max(1, int(100.0 / per_step_ms))
        soak_ms, soak_n = 0.0, 0
        while soak_s > 0 and (soak_ms < soak_s * 1e3 or soak_n < args.steps):
            soak_ms += _timed_steps(chunk, step, stream, flush)
            soak_n += chunk
        # the K timed steps: nothing but the forward in the stream
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ms = _timed_steps(args.steps, step, stream, flush)
        if world > 1:
            dist.barrier()
        # K more steps with the library's per-kernel timing on (an event pair
        # around each lone kernel costs a few microseconds of step time, so it
        # stays out of the K steps above)
        ua.ua_plan_set_profiling(plan.handle, True)
        ua.ua_plan_kernel_times(plan.handle)      # synchronises; nothing recorded yet
        _timed_steps(args.steps, step, stream, flush)
        ktimes = ua.ua_plan_kernel_times(plan.handle)
        ua.ua_plan_set_profiling(plan.handle, False)
        clk.end_load()
    ms_max = max_over_ranks(ms, world, device="cuda")
    soak_max = max_over_ranks(soak_ms / max(soak_n, 1), world, device="cuda")
    step_s = ms_max / 1e3 / args.steps
    job_bytes = sum_over_ranks(byts, world, device="cuda")
    job_flops = sum_over_ranks(flops, world, device="cuda")
    value = _rate(cfg, job_bytes, job_flops, step_s)

    # the whole step against max(bytes / HBM peak, flops / bf16 peak)
    t_bytes, t_flops = byts / (hbm_peak * 1e9), flops / (tf_peak * 1e12)
    step_roof = {"bytes_time_us": t_bytes * 1e6, "flops_time_us": t_flops * 1e6,
                 "bound": "hbm" if t_bytes >= t_flops else "tensor",
                 "frac": max(t_bytes, t_flops) / (ms_max / 1e3 / args.steps)}
    # each kernel's roofline, credited with the work of the sequences the
    # scheduler gave it (host-only schedule of the same batch)
    _, pre_t, dec_t, _ = ua.ua_schedule(b.cu_host, b.kv_host, b.num_q_heads, b.num_kv_heads,
                                        b.head_dim, b.block_size, int(b.block_tables.shape[1]),
                                        kv_dtype=b.kv_dtype, causal=b.causal, window=b.window,
                                        num_splits=args.num_splits, num_sms=info.num_sms)
    mixed = bool(pre_t) and bool(dec_t)
    rooflines = {}
    for kind, tiles in (("prefill", pre_t), ("decode", dec_t)):
        kms, kn = ktimes[kind]
        if not tiles or kn == 0:
            continue
        avg_s = kms / 1e3 / kn
        seqs = sorted({t["seq"] for t in tiles})
        k_bytes = sum(per[s][0] for s in seqs) + (2 * case.num_seqs + 1) * 4
        k_flops = sum(per[s][1] for s in seqs)
        if kind == "prefill":
            ach = k_flops / avg_s / 1e12
            r = {"bound": "tensor", "achieved": ach, "peak": tf_peak, "unit": "TFLOP/s",
                 "frac": ach / tf_peak, "work_per_launch": k_flops}
        else:
            ach = k_bytes / avg_s / 1e9
            r = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                 "frac": ach / hbm_peak, "work_per_launch": k_bytes}
        r["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" \
            if peak_src == "measured" else "fallback"
        if f8p and kind == "prefill":
            r["peak_source"] += " x 2 (e4m3 operands: nominal fp8 / bf16 dense ratio)"
        r["kernel"] = kind
        r["kernel_avg_us"] = avg_s * 1e6
        r["kernel_share"] = kms / max(1e-9, sum(v[0] for v in ktimes.values()))
        r["timing"] = ("device global-timer span, first CTA start to last CTA end (the two "
                       "kernels of a mixed step overlap), over K steps after the timed ones") \
            if mixed else "CUDA events on the launching stream, over K steps after the timed ones"
        # records are per launch configuration: options that change what a
        # launch reads (window, forced splits, CTA count, fp8 products) or its
        # arithmetic (unified max) look up a key of their own
        variant = ("f8p" if f8p and kind == "prefill" else "") + \
            (f"win{args.window}" if args.window else "") + \
            (f"ns{args.num_splits}" if args.num_splits else "") + \
            (f"pc{args.prefill_ctas}" if args.prefill_ctas else "") + \
            ("um" if args.unified_max is not None else "")
        traffic, note, digests = _traffic_record(
            "prefill_wide" if kind == "prefill" and case.head_dim in (192, 256) else kind,
            f"{cfg}{variant}")
        r["traffic"] = traffic
        if note:
            r["traffic_note"] = note
        else:
            r["traffic_digest"] = digests
        rooflines[kind] = r
    # the dominant kernel: the one whose bound is the step's (a mixed step
    # runs both kernels at once), else the only one
    want = "decode" if step_roof["bound"] == "hbm" else "prefill"
    kind = want if want in rooflines else next(iter(rooflines))
    roof = dict(rooflines[kind])
    if len(rooflines) > 1:
        roof["other_kernels"] = {k: v for k, v in rooflines.items() if k != kind}
    launches = sum(v[1] for v in ktimes.values())

    # end to end through the public API with host buffers: one ua_forward_host
    # call per step (scheduling, upload of tiles + lengths + page tables, H2D
    # of q, forward, D2H of the output, synchronisation)
    e2e = None
    if not args.no_e2e:
        q_h = case.q.contiguous().pin_memory()
        cu_h = case.cu_query_lens.to(torch.int32).pin_memory()
        kv_h = case.kv_lens.to(torch.int32).pin_memory()
        bt_h = case.block_tables.to(torch.int32).contiguous().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        tiles_b = 32 * (info.num_prefill_tiles + info.num_decode_tiles) + \
            32 * info.num_combine_groups + 16
        h2d = q_h.numel() * 2 + cu_h.numel() * 4 + kv_h.numel() * 4 + bt_h.numel() * 4 + tiles_b
        d2h = out_h.numel() * 2 + 4
        torch.cuda.synchronize()
        handle = torch.cuda.current_stream().cuda_stream   # the stream every step runs on
        tot = 0.0
        for it in range(args.warmup + args.steps):
            if flush is not None:
                flush.zero_()
                torch.cuda.synchronize()
            t_0 = time.perf_counter()
            err = ua.ua_forward_host(q_h, out_h, cu_h, kv_h, bt_h, b.k_cache, b.v_cache,
                                     b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                     b.num_blocks, b.kv_dtype, b.scale, causal=b.causal,
                                     window=b.window, k_scale=b.k_scale, v_scale=b.v_scale,
                                     num_splits=args.num_splits, stream=handle)
            if it >= args.warmup:
                tot += time.perf_counter() - t_0
            assert err == 0, f"device error word {err}"
        e2e_s = max_over_ranks(tot / args.steps, world, device="cuda")
        e2e = {"value": _rate(cfg, job_bytes, job_flops, e2e_s), "unit": _metric_for(cfg)[1],
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "includes": "one ua_forward_host call per step: CPU scheduling, one upload of "
                           "tiles + lengths + page tables, H2D of q, forward, D2H of the output "
                           "and the error word, stream synchronisation (pinned host buffers)"}
        if args.unified_max is not None or args.prefill_ctas or f8p:
            e2e["note"] = ("the one-call entry point's default settings (no unified max / CTA "
                           "override / fp8 products)")
    plan.close()
    l2_note = ("inputs larger than L2 (%.2f GB > 0.129 GB)" % (byts / 1e9)) if flush is None \
        else "L2 flushed (256 MB write) between timed steps"
    del b, out, flush
    torch.cuda.empty_cache()
    return {
        "workload": WORKLOAD_NAMES[cfg], "metric": _metric_for(cfg)[0], "value": value,
        "unit": _metric_for(cfg)[1], "steps": args.steps, "ms_per_step": ms_max / args.steps,
        "sustained": {"value": _rate(cfg, job_bytes, job_flops, soak_max / 1e3),
                      "ms_per_step": soak_max, "steps": soak_n, "seconds": soak_ms / 1e3}
        if soak_n else None,
        "dtype": "e4m3 Q, K, V, P operands (kind::f8f6f4), fp32 accumulate" if f8p
                 else _dtype_for(case),
        "l2": l2_note,
        "tiles": {"decode": info.num_decode_tiles, "prefill": info.num_prefill_tiles,
                  "split_tokens": info.split_tokens,
                  "prefill_ctas": args.prefill_ctas or info.num_prefill_ctas},
        "algorithmic": {"bytes_per_step": byts, "flops_per_step": flops},
        "pct_of_peak": (value / world) / (tf_peak if cfg in FLOP_CONFIGS else hbm_peak),
        "roofline": roof, "step_roofline": step_roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches), "kernel_ms": {k: v[0] for k, v in ktimes.items()},
        "clocks": clk.summary(),
    }


def run_ours(args):
    import torch
    import torch.distributed as dist
    from paged_kv_attention_unified_gb300 import build as B

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    B.build()
    cfg = args.workload
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    head = measure_attention(cfg, args, rank, world, with_cpu, args.soak, args.cpu_budget)
    if args.per_config == "auto":
        extra = [3, 4, 5] if cfg == 2 and not args.window and not args.num_splits and \
            args.unified_max is None and not args.prefill_ctas and not args.fp8_products else []
    elif args.per_config in ("", "none"):
        extra = []
    else:
        extra = [int(x) for x in args.per_config.split(",") if x]
    per_config = {}
    for c in extra:
        r = measure_attention(c, args, rank, world, with_cpu, args.soak_per_config,
                              args.cpu_budget_per_config)
        per_config[str(c)] = r
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    line = {
        "metric": head["metric"], "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"], "data": "synthetic (seeded N(0,1), random page tables)",
        "config": {"workload": head["workload"], "l2": head["l2"],
                   "parallelism": "replicas: an independent batch per GPU, no collective",
                   "decode_tiles": head["tiles"]["decode"],
                   "prefill_tiles": head["tiles"]["prefill"],
                   "split_tokens": head["tiles"]["split_tokens"],
                   "prefill_ctas": head["tiles"]["prefill_ctas"],
                   **({"unified_max": args.unified_max} if args.unified_max is not None else {}),
                   **({"num_splits": args.num_splits} if args.num_splits else {}),
                   **({"window": args.window} if args.window else {}),
                   **({"fp8_products": True} if args.fp8_products else {})},
        "algorithmic": head["algorithmic"], "pct_of_peak": head["pct_of_peak"],
        "sustained": head["sustained"], "roofline": head["roofline"],
        "step_roofline": head["step_roofline"], "cpu_baseline": head["cpu_baseline"],
        "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
        "kernel_ms": head["kernel_ms"], "clocks": head["clocks"],
    }
    if per_config:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _reference_append(args, case, step_budget):
    """Reference arm of --op append: the oracle's append, rank 0, host cores."""
    import concurrent.futures
    import multiprocessing as mp
    cfg = args.workload
    row = case.num_kv_heads * case.head_dim
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    toks, spent = 0, 0.0
    with concurrent.futures.ProcessPoolExecutor(
            max_workers=1, mp_context=mp.get_context("spawn")) as ex:
        for k in range(args.warmup + args.steps):
            t, sp = ex.submit(_oracle_append_worker, cfg, step_budget).result()
            if k >= args.warmup:
                toks, spent = toks + t, spent + sp
    value = 2 * toks * row * (2 + elt) / spent / 1e9
    sample = (f"each step: the oracle's append over consecutive whole sequences for about "
              f"{step_budget:.1f} s of single-thread work")
    line = {
        "impl": "reference", "metric": "append-KV GB/s (algorithmic new K/V bytes read + cache "
        "bytes written / step time)", "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (CPU oracle)", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": WORKLOAD_NAMES[cfg], "op": "append_kv",
                   "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- append-KV (writing the step's new K/V into the paged cache) ----

def append_work(case):
    """Bytes one append moves: the new K and V rows read (bf16) and written
    (cache element size), plus cu_query_lens, kv_lens and one page-table entry
    per new token."""
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    T = int(case.cu_query_lens[-1])
    row = case.num_kv_heads * case.head_dim
    return 2 * T * row * (2 + elt) + 4 * (2 * case.num_seqs + 1) + 4 * T


def _new_kv(case, seed=1):
    import torch
    g = torch.Generator().manual_seed(seed)
    T = int(case.cu_query_lens[-1])
    shape = (T, case.num_kv_heads, case.head_dim)
    return (torch.randn(shape, generator=g).to(torch.bfloat16),
            torch.randn(shape, generator=g).to(torch.bfloat16))


def _oracle_append_worker(cfg, budget_s):
    """Spawned process, one thread: the oracle's append over consecutive
    sequences of the workload for about budget_s. Returns (tokens, seconds)."""
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import numpy as np
    import oracle
    import workloads as W
    case = W.CONFIGS[cfg]()
    r = case.raw()
    kn, vn = _new_kv(case)
    kn = kn.view(__import__("torch").int16).numpy().view(np.uint16)
    vn = vn.view(__import__("torch").int16).numpy().view(np.uint16)
    cu = r["cu_query_lens"]
    toks, spent, s = 0, 0.0, 0
    while spent < budget_s and s < case.num_seqs:
        t0 = time.perf_counter()
        oracle.append_kv(kn[cu[s]:cu[s + 1]], vn[cu[s]:cu[s + 1]], r["k_cache"], r["v_cache"],
                         [0, int(cu[s + 1] - cu[s])], r["kv_lens"][s:s + 1],
                         r["block_tables"][s:s + 1], case.block_size, kv_dtype=case.kv_dtype,
                         k_scale=case.k_scale, v_scale=case.v_scale)
        spent += time.perf_counter() - t0
        toks += int(cu[s + 1] - cu[s])
        s += 1
    return toks, spent


def run_append(args):
    """One step = ua_append_kv of every new token of the workload's batch (the
    q tokens' K and V) into its paged cache; HBM-bound."""
    import torch
    import concurrent.futures
    import multiprocessing as mp
    import paged_kv_attention_unified_gb300 as ua
    from paged_kv_attention_unified_gb300 import build as B
    from paged_kv_attention_unified_gb300 import torch_utils as tu
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    B.build()
    cfg = args.workload
    case = rank_case(cfg, rank)
    byts = append_work(case)
    hbm_peak, _, peak_src = _peaks()
    T = int(case.cu_query_lens[-1])
    row = case.num_kv_heads * case.head_dim
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        with concurrent.futures.ProcessPoolExecutor(
                max_workers=1, mp_context=mp.get_context("spawn")) as ex:
            toks, spent = ex.submit(_oracle_append_worker, cfg, args.cpu_budget).result()
        cpu_b = 2 * toks * row * (2 + elt)
        cpu = {"value": cpu_b / spent / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{toks} of {T} new tokens (whole sequences), {spent:.1f} s of "
                         "single-thread fp64-oracle work"}
    b = tu.to_device(case)
    kn, vn = (t.cuda() for t in _new_kv(case))
    plan = tu.make_plan(b)
    ua.ua_plan_set_profiling(plan.handle, True)
    for _ in range(args.warmup):
        tu.append_kv(plan, b, kn, vn)
    torch.cuda.synchronize()
    ua.ua_plan_kernel_times(plan.handle)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ms = 0.0
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.steps):
            flush.zero_()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            tu.append_kv(plan, b, kn, vn)
            t1.record(stream)
            torch.cuda.synchronize()
            ms += t0.elapsed_time(t1)
    kt = ua.ua_plan_kernel_times(plan.handle)["append"]
    ms_max = max_over_ranks(ms, world, device="cuda")
    job_bytes = sum_over_ranks(byts, world, device="cuda")
    value = job_bytes / (ms_max / 1e3 / args.steps) / 1e9
    avg_s = kt[0] / 1e3 / max(1, kt[1])
    ach = byts / avg_s / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
            "frac": ach / hbm_peak, "work_per_launch": byts, "kernel": "append",
            "kernel_avg_us": avg_s * 1e6, "kernel_share": 1.0,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured"
            else "fallback",
            "traffic": _traffic_record("append", cfg)[0]}
    # end to end: pinned host K/V rows -> device, append, read the error word
    kh, vh = kn.cpu().pin_memory(), vn.cpu().pin_memory()
    tot = 0.0
    for it in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t_0 = time.perf_counter()
        kn.copy_(kh, non_blocking=True)
        vn.copy_(vh, non_blocking=True)
        tu.append_kv(plan, b, kn, vn)
        err = plan.last_device_error()
        if it >= args.warmup:
            tot += time.perf_counter() - t_0
    assert err == 0
    plan.close()
    if rank != 0:
        return 0
    line = {
        "metric": "append-KV GB/s (algorithmic new K/V bytes read + cache bytes written / step time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 -> fp8 e4m3 (x / scale, saturating)" if elt == 1 else "bf16 copy",
        "data": "synthetic (seeded N(0,1), random page tables)",
        "config": {"workload": WORKLOAD_NAMES[cfg], "op": "append_kv", "new_tokens": T,
                   "l2": "L2 flushed (256 MB write) between timed steps",
                   "parallelism": "replicas: an independent batch per GPU, no collective"},
        "algorithmic": {"bytes_per_step": byts},
        "pct_of_peak": (value / world) / hbm_peak,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": byts / (tot / args.steps) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(kh.numel() * 2 * 2), "d2h_bytes_per_step": 4,
                "includes": "H2D of the new K/V rows, append, read of the error word"},
        "gpu_launches": int(kt[1]), "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="wall seconds of the oracle on every host core for the headline "
                         "workload's cpu_baseline")
    ap.add_argument("--cpu-budget-per-config", type=float, default=4.0)
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of back-to-back steps before the K timed steps (sustained "
                         "rate and clock record under load)")
    ap.add_argument("--soak-per-config", type=float, default=0.5)
    ap.add_argument("--per-config", default="auto",
                    help="comma-separated workloads measured after the headline one and "
                         "reported under per_config (auto: 3,4,5 after the default workload 2; "
                         "none: only the headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", default="attention", choices=["attention", "append"],
                    help="attention: the forward step (default); append: ua_append_kv of the "
                         "step's new K/V")
    ap.add_argument("--window", type=int, default=0, metavar="W",
                    help="left sliding window of W keys for the attention step (0: none)")
    ap.add_argument("--num-splits", type=int, default=0, metavar="N",
                    help="cut every decode tile into N split pieces (0: automatic sizing)")
    ap.add_argument("--fp8-products", action="store_true",
                    help="fp8 cache workloads: prefill tiles with e4m3 tensor-core products "
                         "(ua_plan_set_fp8_products)")
    ap.add_argument("--prefill-ctas", type=int, default=0, metavar="P",
                    help="persistent prefill CTAs of a mixed step (0: the scheduler's choice)")
    ap.add_argument("--unified-max", type=float, default=None, metavar="PHI",
                    help="decode rows start from the unified max PHI (scaled-score units) "
                         "instead of their first maximum (off by default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "append":
        return run_append(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
